// kernels_compress.cu -- persistent tcgen05 compress kernel of the MAPL codec.
//
// MAPL §3.2 eq. (1), with the anchor folded through M = P_send A:
//     Z = X A - E_send[tids] M                  (one TMEM accumulation per tile)
// followed, with VQ, by the multi-codebook residual quantisation of §3.5: for
// every group g and round rho the nearest code of the group's residual.
//
// One CTA per SM loops over 128-token tiles.  Warp roles (12 warps):
//   warp 0  lane 0: TMA producer.  A ring of shared-memory stages carries, in
//                   order, the projection items of tile k (X block + A^T block,
//                   then -M^T split blocks with their gathered anchor rows)
//                   and the codebook tiles of tile k-1's VQ.
//   warp 1        : TMEM allocation; lane 0 issues every tcgen05.mma of the
//                   CTA: the projection MMAs (into one of two Z accumulators,
//                   double buffered across tiles) and the VQ distance MMAs,
//                   interleaved by non-blocking barrier probes.
//   warps 2, 3    : idle.
//   warps 4..11   : epilogue.  Warp w reads TMEM lanes 32*(w%4)..+31 (token
//                   rows); warps 4..7 scan codes [0, K/2), warps 8..11 codes
//                   [K/2, K) of the same rows.  Group g's residual is owned by
//                   the half (g & 1) warp of each quadrant.
//
// VQ decision.  The residual u (fp32, kept in the Z accumulator's columns) is
// split into u_hi = bf16(u), u_lo = bf16(u - u_hi) and one MMA per half gives
// s_k = u_hi.c_k + u_lo.c_k for all codes (|s_k - u.c_k| <= ~2^-18 |u||c_k|
// plus fp32 accumulation).  D~_k = ||c_k||^2 - 2 s_k is scanned for the best
// and second best; when the two are within twice the certified error bound
// every code inside that band is re-scored with the exact squared distance in
// fp64.  The chosen index is therefore the exact nearest code of the fp32
// residual (lowest index on exact ties).  The residual update is fp32.
//
// Every wait is time bounded (mbar_wait); a CTA that gives up sets the device
// error word and unwinds through its common exit.
#include "mapl_internal.h"
#include "ptx.cuh"

namespace mapl {

namespace {

constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kMaxStages = 8;
constexpr int kNSlot = 4;                       // residual operand slots (groups in flight)
constexpr uint32_t kBlockBytes = kTile * 128;   // 128 rows x 64 bf16, 128B swizzled
constexpr uint32_t kFull = 0xffffffffu;

struct Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t zfull[2];
  uint64_t zempty[2];
  uint64_t uready[kNSlot];
  uint64_t dfull[2];
  uint64_t dempty[2];
  uint64_t pair[4];                 // the two epilogue warps of a TMEM quadrant
  uint32_t tmem_base;
  int abort;
  float xb1[2][2][kTile];           // [item parity][half][row] best of a half
  float xb2[2][2][kTile];           // second best of a half
  int xk1[2][2][kTile];             // index of the best
  float nu[kNSlot][2][kTile];       // ||u|| of the residual in a slot [round parity]
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

__device__ __forceinline__ void give_up(Ctl* ctl, int* err) {
  ctl->abort = 1;
  atomicOr(err, kErrTimeout);
}

// Position of an item in the producer's order (P = projection items of a
// tile, V = VQ codebook items of a tile).  With two Z accumulators the next
// tile's projection runs ahead of this tile's VQ: P0, P1, V0, P2, V1, ...,
// V_{L-1}.  With one accumulator the next projection must wait for this
// tile's VQ, so its items may not block the ring: P0, V0, P1, V1, ...
__device__ __forceinline__ int base_P(int it, int nP, int nV, int nzb) {
  if (nzb == 1) return it * (nP + nV);
  return it == 0 ? 0 : nP + (it - 1) * (nP + nV);
}
__device__ __forceinline__ int base_V(int it, int L, int nP, int nV, int nzb) {
  if (nzb == 1) return it * (nP + nV) + nP;
  if (it < L - 1) return base_P(it + 1, nP, nV, nzb) + nP;
  return L == 1 ? nP : base_P(it, nP, nV, nzb) + nP + nV;
}

struct Geo {
  int r, nkx, nkr, na, nP, nV, nh, nrow, GD, B, nzb, zstride;
};

__device__ __forceinline__ Geo geometry(const CompressArgs& a, bool vq) {
  Geo g;
  g.r = a.r;
  g.nkx = a.d / 64;
  g.nkr = a.r / 64;
  g.na = kNumSplit * g.nkr;
  g.nP = g.nkx + g.na;
  g.nV = vq ? a.G * a.R : 0;
  g.nh = a.r > 256 ? 2 : 1;
  g.nrow = a.r > 256 ? 256 : a.r;
  g.GD = a.gd;
  g.B = a.G < kNSlot ? a.G : kNSlot;
  g.nzb = vq ? (a.r <= 128 ? 2 : 1) : (2 * a.r <= 512 ? 2 : 1);
  g.zstride = a.r;
  return g;
}

// Bounded wait on an mbarrier by all lanes of a warp; false (for every lane)
// if any lane gave up.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, Ctl* ctl,
                                          uint64_t budget) {
  const bool ok = mbar_wait(bar, parity, &ctl->abort, budget);
  return __all_sync(kFull, ok);
}

// Pair sync of the two epilogue warps of quadrant q (mbarrier of count 2,
// one arrival per warp).  Lanes' shared-memory writes before the call are
// visible to the partner warp after it.
__device__ __forceinline__ bool pair_sync(Ctl* ctl, int q, int lane, uint32_t& cnt,
                                          uint64_t budget) {
  __threadfence_block();
  __syncwarp();
  const uint32_t bar = smem_u32(&ctl->pair[q]);
  if (lane == 0) mbar_arrive(bar);
  const bool ok = warp_wait(bar, cnt & 1u, ctl, budget);
  ++cnt;
  return ok;
}

template <int GD>
__device__ __forceinline__ void tmem_load_group(uint32_t taddr, float (&u)[GD]) {
#pragma unroll
  for (int c = 0; c < GD; c += 16) {
    float t[16];
    tmem_ld16(taddr + c, t);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) u[c + i] = t[i];
  }
}

template <int GD>
__device__ __forceinline__ void tmem_store_group(uint32_t taddr, const float (&u)[GD]) {
#pragma unroll
  for (int c = 0; c < GD; c += 16) {
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = u[c + i];
    tmem_st16(taddr + c, t);
  }
  tmem_wait_st();
}

// Two-term bf16 split of the residual into the swizzled A operand of the
// distance MMA: row `row` holds [hi (GD) | lo (GD)].
template <int GD>
__device__ __forceinline__ float write_operand(uint32_t slot, int row, const float (&u)[GD]) {
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < GD / 8; ++c) {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x0 = u[c * 8 + 2 * e], x1 = u[c * 8 + 2 * e + 1];
      s = fmaf(x0, x0, s);
      s = fmaf(x1, x1, s);
      const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
      const float2 hf = __bfloat1622float2(h);
      const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
      hw[e] = *reinterpret_cast<const uint32_t*>(&h);
      lw[e] = *reinterpret_cast<const uint32_t*>(&l);
    }
    st_shared_v4(slot + sw128_off(row, c), make_uint4(hw[0], hw[1], hw[2], hw[3]));
    st_shared_v4(slot + sw128_off(row, GD / 8 + c), make_uint4(lw[0], lw[1], lw[2], lw[3]));
  }
  return sqrtf(s) * 1.000001f;
}

// Best / second best of D~_k = ||c_k||^2 - 2 s_k over KH columns of TMEM
// (two interleaved trackers; exact ties keep the lowest index).
__device__ __forceinline__ void scan_half(uint32_t tdist, const float* __restrict__ cn, int KH,
                                          int koff, float& b1, float& b2, int& k1) {
  const float inf = __int_as_float(0x7f800000);
  float a1 = inf, a2 = inf, c1 = inf, c2 = inf;
  int ka = 0, kc = 0;
  for (int c0 = 0; c0 < KH; c0 += 32) {
    float v[32];
    tmem_ld32(tdist + c0, v);
    float cv[32];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(cn + c0) + q);
      cv[4 * q] = f.x;
      cv[4 * q + 1] = f.y;
      cv[4 * q + 2] = f.z;
      cv[4 * q + 3] = f.w;
    }
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float D0 = fmaf(-2.f, v[j], cv[j]);
      const float D1 = fmaf(-2.f, v[j + 1], cv[j + 1]);
      a2 = fminf(a2, fmaxf(a1, D0));
      ka = D0 < a1 ? (koff + c0 + j) : ka;
      a1 = fminf(a1, D0);
      c2 = fminf(c2, fmaxf(c1, D1));
      kc = D1 < c1 ? (koff + c0 + j + 1) : kc;
      c1 = fminf(c1, D1);
    }
  }
  const bool take_c = c1 < a1 || (c1 == a1 && kc < ka);
  b1 = take_c ? c1 : a1;
  k1 = take_c ? kc : ka;
  b2 = fminf(fminf(a2, c2), fmaxf(a1, c1));
}

template <int GD>
__device__ void epilogue_vq(const CompressArgs& a, const Geo& geo, Ctl* ctl, uint32_t tbase,
                            uint32_t ubase, int tile, int zb, int q, int h, int lane,
                            uint32_t& dcnt, uint32_t& pcnt, bool& alive) {
  const int row = q * 32 + lane;
  const int n = tile * kTile + row;
  const bool store = n < a.N;
  bool bad = false;
  if (store) {
    const int t = a.tids[n];
    bad = t < 0 || t >= a.V;
  }
  const uint32_t lanebase = static_cast<uint32_t>(q * 32) << 16;
  const uint32_t tz = tbase + lanebase + zb * geo.zstride;
  const int G = a.G, R = a.R, K = a.K, KH = a.K / 2;
  uint8_t* idx_out = reinterpret_cast<uint8_t*>(a.out) + static_cast<size_t>(n) * R * G;
  const uint64_t bud = a.timeout_ns;

  for (int b0 = 0; b0 < G && alive; b0 += geo.B) {
    const int b1g = b0 + geo.B < G ? b0 + geo.B : G;
    // round-0 operands of the groups this half owns
    for (int g = b0; g < b1g; ++g) {
      if ((g & 1) != h && G > 1) continue;
      if (G == 1 && h == 1) continue;
      float u[GD];
      tmem_load_group<GD>(tz + g * GD, u);
      const int slot = g - b0;
      const float nu = write_operand<GD>(ubase + slot * kBlockBytes, row, u);
      ctl->nu[slot][0][row] = nu;
      fence_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->uready[slot]));
    }
    for (int rho = 0; rho < R && alive; ++rho) {
      for (int g = b0; g < b1g && alive; ++g) {
        const int slot = g - b0;
        const int book = rho * G + g;
        const bool owner = (G == 1) ? (h == 0) : ((g & 1) == h);
        const int par = static_cast<int>(dcnt & 1u);
        // 1. distances of this half are in TMEM
        if (!warp_wait(smem_u32(&ctl->dfull[h]), dcnt & 1u, ctl, bud)) {
          give_up(ctl, a.err);
          alive = false;
          break;
        }
        tc_fence_after();
        const uint32_t tdist = tbase + lanebase + 256 + h * 128;
        float b1, b2;
        int k1;
        scan_half(tdist, a.cnorm + static_cast<size_t>(book) * K + h * KH, KH, h * KH, b1, b2, k1);
        ctl->xb1[par][h][row] = b1;
        ctl->xb2[par][h][row] = b2;
        ctl->xk1[par][h][row] = k1;
        if (!pair_sync(ctl, q, lane, pcnt, bud)) {
          give_up(ctl, a.err);
          alive = false;
          break;
        }
        // 2. merge the two halves (half 0 holds the lower indices)
        const float ob1 = ctl->xb1[par][h ^ 1][row];
        const float ob2 = ctl->xb2[par][h ^ 1][row];
        const int ok1 = ctl->xk1[par][h ^ 1][row];
        const bool take_o = ob1 < b1 || (ob1 == b1 && ok1 < k1);
        const float B1 = take_o ? ob1 : b1;
        int K1 = take_o ? ok1 : k1;
        const float B2 = fminf(fminf(b2, ob2), fmaxf(b1, ob1));
        const float nu = ctl->nu[slot][rho & 1][row];
        const float cm = __ldg(a.cmax + book);
        // certified bound on |D~_k - D_k| (two-term split, fp32 accumulation
        // of 2*GD exact products, fp32 rounding of ||c||^2 and the fma)
        const float eps = 2e-5f * nu * cm + 1.2e-7f * (cm * cm + 2.f * nu * cm + fabsf(B1));
        const bool need = (B2 - B1) <= 2.f * eps;
        float u[GD];
        bool have_u = false;
        if (__any_sync(kFull, need)) {
          if (owner) {
            tmem_load_group<GD>(tz + g * GD, u);
            have_u = true;
            const float thr = B1 + 2.f * eps;
            double best = 1e300;
            int kb = K1;
            for (int hh = 0; hh < 2; ++hh) {
              const uint32_t td = tbase + lanebase + 256 + hh * 128;
              const float* cnh = a.cnorm + static_cast<size_t>(book) * K + hh * KH;
              for (int c0 = 0; c0 < KH; c0 += 16) {
                float v[16];
                __syncwarp();
                tmem_ld16(td + c0, v);
                tmem_wait_ld();
                if (!need) continue;
                for (int j = 0; j < 16; ++j) {
                  if (fmaf(-2.f, v[j], __ldg(cnh + c0 + j)) > thr) continue;
                  const int kk = hh * KH + c0 + j;
                  const __nv_bfloat16* cr = a.Cb + (static_cast<size_t>(book) * K + kk) * GD;
                  double e = 0.0;
#pragma unroll
                  for (int i = 0; i < GD; ++i) {
                    const double df = static_cast<double>(u[i]) -
                                      static_cast<double>(__bfloat162float(cr[i]));
                    e = fma(df, df, e);
                  }
                  if (e < best) {
                    best = e;
                    kb = kk;
                  }
                }
              }
            }
            if (need) K1 = kb;
          }
          // the partner keeps its half until the owner has re-read it
          if (!pair_sync(ctl, q, lane, pcnt, bud)) {
            give_up(ctl, a.err);
            alive = false;
            break;
          }
        }
        // 3. release this half's distance buffer
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->dempty[h]));
        ++dcnt;
        if (!owner) continue;
        // 4. owner: record the index, update the residual, next operand
        if (store) idx_out[rho * G + g] = bad ? static_cast<uint8_t>(0) : static_cast<uint8_t>(K1);
        if (rho + 1 < R) {
          if (!have_u) tmem_load_group<GD>(tz + g * GD, u);
          const uint4* cr4 =
              reinterpret_cast<const uint4*>(a.Cb + (static_cast<size_t>(book) * K + K1) * GD);
#pragma unroll
          for (int c = 0; c < GD / 8; ++c) {
            const uint4 w = __ldg(cr4 + c);
            const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(hp[e]);
              u[c * 8 + 2 * e] -= f.x;
              u[c * 8 + 2 * e + 1] -= f.y;
            }
          }
          tmem_store_group<GD>(tz + g * GD, u);
          const float nn = write_operand<GD>(ubase + slot * kBlockBytes, row, u);
          ctl->nu[slot][(rho + 1) & 1][row] = nn;
          fence_async_shared();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctl->uready[slot]));
        }
      }
    }
  }
}

template <int GD>
__global__ void __launch_bounds__(kThreads, 1)
    k_compress(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmAt,
               const __grid_constant__ CUtensorMap tmMt, const __grid_constant__ CUtensorMap tmC,
               const __grid_constant__ CUtensorMap tmE, const CompressArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  const bool vq = a.mode == kModeVQ;
  const Geo geo = geometry(a, vq);
  const int nst = a.nstage;
  const uint32_t sb = a.stage_bytes;
  const uint32_t ring = smem_u32(base);
  const uint32_t ubase = ring + nst * sb;
  const uint32_t ubytes = vq ? geo.B * kBlockBytes : 0u;
  Ctl* ctl = reinterpret_cast<Ctl*>(base + nst * sb + ubytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = (a.N + kTile - 1) / kTile;
  // tiles of this CTA: blockIdx.x, blockIdx.x + gridDim.x, ...
  const int L = blockIdx.x < ntiles ? (ntiles - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
  uint32_t tmem_cols = 32;
  {
    const uint32_t need = vq ? 512u : static_cast<uint32_t>(geo.nzb * geo.r);
    while (tmem_cols < need) tmem_cols <<= 1;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int z = 0; z < 2; ++z) {
      mbar_init(smem_u32(&ctl->zfull[z]), 1);
      mbar_init(smem_u32(&ctl->zempty[z]), 8);
      mbar_init(smem_u32(&ctl->dfull[z]), 1);
      mbar_init(smem_u32(&ctl->dempty[z]), 4);
    }
    for (int s = 0; s < kNSlot; ++s) mbar_init(smem_u32(&ctl->uready[s]), 4);
    for (int p = 0; p < 4; ++p) mbar_init(smem_u32(&ctl->pair[p]), 2);
    ctl->abort = 0;
    fence_mbar_init();
    fence_async_shared();
  }
  if (warp == 1) tmem_alloc(smem_u32(&ctl->tmem_base), tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ctl->tmem_base;
  const uint64_t bud = a.timeout_ns;

  if (warp == 0 && lane == 0) {
    // --------------------------------------------------------------- producer
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmAt);
    prefetch_tmap(&tmMt);
    prefetch_tmap(&tmE);
    if (vq) prefetch_tmap(&tmC);
    int i = 0;
    bool ok = true;
    auto acquire = [&](uint32_t& st, uint32_t& fb) -> bool {
      const int s = i % nst, use = i / nst;
      if (!mbar_wait(smem_u32(&ctl->empty[s]), (use & 1) ^ 1, &ctl->abort, bud)) return false;
      st = ring + s * sb;
      fb = smem_u32(&ctl->full[s]);
      return true;
    };
    for (int k = 0; k <= L && ok; ++k) {
      // tile whose VQ codebooks follow this iteration's projection items
      const int kv = geo.nzb == 1 ? k : k - 1;
      if (k < L) {
        const int tile = blockIdx.x + k * gridDim.x;
        for (int p = 0; p < geo.nP && ok; ++p, ++i) {
          uint32_t st, fb;
          if (!(ok = acquire(st, fb))) break;
          if (p < geo.nkx) {
            mbar_arrive_expect_tx(fb, kBlockBytes + geo.r * 128u);
            tma_load_2d(st, &tmX, p * 64, tile * kTile, fb);
            for (int hh = 0; hh < geo.nh; ++hh)
              tma_load_2d(st + kBlockBytes + hh * 256u * 128u, &tmAt, p * 64, hh * 256, fb);
          } else {
            const int j = p - geo.nkx, sp = j / geo.nkr, kb = j % geo.nkr;
            mbar_arrive_expect_tx(fb, kBlockBytes + geo.r * 128u);
            for (int hh = 0; hh < geo.nh; ++hh)
              tma_load_2d(st + kBlockBytes + hh * 256u * 128u, &tmMt, kb * 64,
                          sp * geo.r + hh * geo.nrow, fb);
            // anchor rows E[tids] of the tile (invalid ids and rows past N
            // read row 0; their outputs are zeroed by the epilogue)
            for (int q4 = 0; q4 < kTile / 4; ++q4) {
              int rr[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int n = tile * kTile + q4 * 4 + e;
                int t = n < a.N ? __ldg(a.tids + n) : 0;
                rr[e] = (t < 0 || t >= a.V) ? 0 : t;
              }
              tma_gather4(st + q4 * 512, &tmE, kb * 64, rr[0], rr[1], rr[2], rr[3], fb);
            }
          }
        }
      }
      if (kv >= 0 && kv < L && vq && ok) {
        // codebook tiles of tile kv, in the epilogue's item order
        for (int b0 = 0; b0 < a.G && ok; b0 += geo.B) {
          const int b1g = b0 + geo.B < a.G ? b0 + geo.B : a.G;
          for (int rho = 0; rho < a.R && ok; ++rho)
            for (int g = b0; g < b1g && ok; ++g, ++i) {
              uint32_t st, fb;
              if (!(ok = acquire(st, fb))) break;
              mbar_arrive_expect_tx(fb, a.K * 128u);
              tma_load_2d(st, &tmC, 0, (rho * a.G + g) * a.K, fb);
            }
        }
      }
    }
    if (!ok) give_up(ctl, a.err);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    // One thread issues every tcgen05 operation of the CTA.  It interleaves
    // two independent streams with non-blocking probes: the VQ distance MMAs
    // of the tile in the epilogue (first, they gate the epilogue) and the
    // projection MMAs of the next tile.
    const uint32_t idz = idesc_bf16(kTile, geo.nrow);
    const int KH = vq ? a.K / 2 : 16;
    const uint32_t idd = idesc_bf16(kTile, KH);
    // projection stream
    int pj_it = 0, pj_p = 0;
    bool pj_started = false;
    // VQ stream: item (b0, rho, g) of tile vq_it, half vq_hh
    int vq_it = 0, vq_b0 = 0, vq_rho = 0, vq_g = 0, vq_hh = 0, vq_i = 0;
    bool vq_u = false, vq_c = false;
    uint32_t ucnt[kNSlot] = {0u, 0u, 0u, 0u};
    uint32_t e = 0;
    // Ring uses of each stage observed so far.  The two streams consume
    // interleaved items of one ring; a probe of use u of a stage is only
    // meaningful once use u-1 was consumed (a parity probe cannot tell
    // phase u from phase u-2), so each stream waits for its turn first.
    int seen[kMaxStages];
    for (int q = 0; q < kMaxStages; ++q) seen[q] = 0;
    if (vq && L > 0) vq_i = base_V(0, L, geo.nP, geo.nV, geo.nzb);
    const int vq_end = vq ? L : 0;
    uint64_t last = global_ns();
    uint32_t idle = 0;
    bool ok = true;
    while (ok && (pj_it < L || vq_it < vq_end)) {
      bool progressed = false;
      if (vq_it < vq_end) {
        const int b1g = vq_b0 + geo.B < a.G ? vq_b0 + geo.B : a.G;
        const int slot = vq_g - vq_b0;
        const int s = vq_i % nst, use = vq_i / nst;
        if (!vq_u && mbar_test(smem_u32(&ctl->uready[slot]), ucnt[slot] & 1u)) {
          vq_u = true;
          ++ucnt[slot];
        }
        if (vq_u && !vq_c && seen[s] == use && mbar_test(smem_u32(&ctl->full[s]), use & 1)) {
          vq_c = true;
          ++seen[s];
        }
        if (vq_u && vq_c && mbar_test(smem_u32(&ctl->dempty[vq_hh]), (e & 1u) ^ 1u)) {
          tc_fence_after();
          const uint32_t st = ring + s * sb;
          const uint32_t us = ubase + slot * kBlockBytes;
#pragma unroll
          for (int k = 0; k < 2 * (GD > 0 ? GD : 16) / 16; ++k)
            mma_bf16(tbase + 256 + vq_hh * 128, sw128_desc(us + k * 32),
                     sw128_desc(st + vq_hh * KH * 128u + k * 32), idd, k != 0 ? 1u : 0u);
          mma_commit(smem_u32(&ctl->dfull[vq_hh]));
          progressed = true;
          if (vq_hh == 0) {
            vq_hh = 1;
          } else {
            mma_commit(smem_u32(&ctl->empty[s]));
            vq_hh = 0;
            vq_u = vq_c = false;
            ++e;
            ++vq_i;
            if (++vq_g == b1g) {
              vq_g = vq_b0;
              if (++vq_rho == a.R) {
                vq_rho = 0;
                vq_b0 += geo.B;
                vq_g = vq_b0;
                if (vq_b0 >= a.G) {
                  vq_b0 = vq_g = 0;
                  if (++vq_it < L) vq_i = base_V(vq_it, L, geo.nP, geo.nV, geo.nzb);
                }
              }
            }
          }
        }
      }
      if (pj_it < L) {
        const int zb = geo.nzb == 2 ? (pj_it & 1) : 0;
        const int zuse = geo.nzb == 2 ? (pj_it >> 1) : pj_it;
        if (!pj_started && mbar_test(smem_u32(&ctl->zempty[zb]), (zuse & 1) ^ 1)) {
          pj_started = true;
          tc_fence_after();
        }
        if (pj_started) {
          const int i = base_P(pj_it, geo.nP, geo.nV, geo.nzb) + pj_p;
          const int s = i % nst, use = i / nst;
          if (seen[s] == use && mbar_test(smem_u32(&ctl->full[s]), use & 1)) {
            ++seen[s];
            tc_fence_after();
            const uint32_t st = ring + s * sb;
            const uint32_t dz = tbase + zb * geo.zstride;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = sw128_desc(st + k * 32);
              for (int hh = 0; hh < geo.nh; ++hh)
                mma_bf16(dz + hh * 256, ad,
                         sw128_desc(st + kBlockBytes + hh * 256u * 128u + k * 32), idz,
                         (pj_p | k) != 0 ? 1u : 0u);
            }
            mma_commit(smem_u32(&ctl->empty[s]));
            progressed = true;
            if (++pj_p == geo.nP) {
              mma_commit(smem_u32(&ctl->zfull[zb]));
              pj_p = 0;
              pj_started = false;
              ++pj_it;
            }
          }
        }
      }
      if (progressed) {
        idle = 0;
        continue;
      }
      if ((++idle & 63u) == 0u) {
        const uint64_t now = global_ns();
        if (idle == 64u) last = now;
        if (ctl->abort || now - last > bud) ok = false;
      }
    }
    if (!ok) give_up(ctl, a.err);
  } else if (warp >= kEpiWarp0) {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3, h = (warp - kEpiWarp0) >> 2;
    uint32_t dcnt = 0, pcnt = 0;
    bool alive = true;
    for (int it = 0; it < L && alive; ++it) {
      const int tile = blockIdx.x + it * gridDim.x;
      const int zb = geo.nzb == 2 ? (it & 1) : 0;
      const int zuse = geo.nzb == 2 ? (it >> 1) : it;
      if (!warp_wait(smem_u32(&ctl->zfull[zb]), zuse & 1, ctl, bud)) {
        give_up(ctl, a.err);
        break;
      }
      tc_fence_after();
      if (vq) {
        if constexpr (GD > 0)
          epilogue_vq<GD>(a, geo, ctl, tbase, ubase, tile, zb, q, h, lane, dcnt, pcnt, alive);
      } else {
        const int row = q * 32 + lane;
        const int n = tile * kTile + row;
        const bool store = n < a.N;
        bool bad = false;
        if (store) {
          const int t = a.tids[n];
          bad = t < 0 || t >= a.V;
          if (bad) atomicOr(a.err, kErrBadToken);
        }
        const uint32_t tz = tbase + (static_cast<uint32_t>(q * 32) << 16) + zb * geo.zstride;
        const int half = geo.r / 2;
        for (int c0 = h * half; c0 < (h + 1) * half; c0 += 32) {
          float v[32];
          __syncwarp();
          tmem_ld32(tz + c0, v);
          tmem_wait_ld();
          if (bad) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.f;
          }
          if (!store) continue;
          if (a.mode == kModeZ32) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) +
                                                    static_cast<size_t>(n) * geo.r + c0);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) +
                                                  static_cast<size_t>(n) * geo.r + c0);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]),
                                  pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                                  pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                                  pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
          }
        }
      }
      if (vq && alive) {
        // flag invalid token ids once per row (owner-independent)
        const int n = tile * kTile + q * 32 + lane;
        if (h == 0 && n < a.N) {
          const int t = a.tids[n];
          if (t < 0 || t >= a.V) atomicOr(a.err, kErrBadToken);
        }
      }
      if (!alive) break;
      // release the Z accumulator of this tile
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->zempty[zb]));
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

template <typename KernelT>
cudaError_t set_smem(KernelT k, uint32_t bytes) {
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

}  // namespace

uint32_t compress_ctl_bytes() { return static_cast<uint32_t>(sizeof(Ctl)); }

cudaError_t launch_compress_tc(const CUtensorMap& tmX, const CUtensorMap& tmAt,
                               const CUtensorMap& tmMt, const CUtensorMap& tmC,
                               const CUtensorMap& tmE, const CompressArgs& a,
                               uint32_t smem_bytes, int grid, cudaStream_t s) {
  cudaError_t e;
  switch (a.mode == kModeVQ ? a.gd : 0) {
    case 0:
      e = set_smem(k_compress<0>, smem_bytes);
      if (e != cudaSuccess) return e;
      k_compress<0><<<grid, kThreads, smem_bytes, s>>>(tmX, tmAt, tmMt, tmC, tmE, a);
      break;
    case 16:
      e = set_smem(k_compress<16>, smem_bytes);
      if (e != cudaSuccess) return e;
      k_compress<16><<<grid, kThreads, smem_bytes, s>>>(tmX, tmAt, tmMt, tmC, tmE, a);
      break;
    case 32:
      e = set_smem(k_compress<32>, smem_bytes);
      if (e != cudaSuccess) return e;
      k_compress<32><<<grid, kThreads, smem_bytes, s>>>(tmX, tmAt, tmMt, tmC, tmE, a);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace mapl
