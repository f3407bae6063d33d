// kernels_compress.cu -- persistent tcgen05 compress kernel of the MAPL codec.
//
// MAPL §3.2 eq. (1), with the anchor folded through M = P_send A:
//     Z = X A - E_send[tids] M                  (one TMEM accumulation per tile)
// followed, with VQ, by the multi-codebook residual quantisation of §3.5: for
// every group g and round rho the nearest code of the group's residual.
//
// One CTA per SM loops over 128-token tiles.  Warp roles (12 warps):
//   warp 0  lane 0: TMA producer of the main ring: per tile, X blocks with A^T
//                   blocks, then -M^T split blocks with the tile's anchor rows
//                   E[tids] (tile::gather4).
//   warp 2  lane 0: TMA producer of a 2-stage codebook ring (VQ only).
//   warp 1        : TMEM allocation; lane 0 issues every tcgen05.mma of the
//                   CTA: the projection MMAs (into one of two Z accumulators,
//                   double buffered across tiles) and the VQ distance MMAs,
//                   interleaved by non-blocking barrier probes.
//   warp 3        : idle.
//   warps 4..11   : epilogue.  Warp w reads TMEM lanes 32*(w%4)..+31 (token
//                   rows); warps 4..7 scan codes [0, K/2), warps 8..11 codes
//                   [K/2, K) of the same rows.  Group g's residual is owned by
//                   the half (g & 1) warp of each quadrant.
//
// VQ decision.  The residual u (fp32, kept in the Z accumulator's columns) is
// split into u_hi = bf16(u), u_lo = bf16(u - u_hi) and one N = K MMA gives
// s_k = u_hi.c_k + u_lo.c_k for all codes (|s_k - u.c_k| <= ~2^-18 |u||c_k|
// plus fp32 accumulation).  D~_k = ||c_k||^2 - 2 s_k is scanned for the best
// and second best; when the two are within twice the certified error bound
// every code inside that band is re-scored with the squared distance in
// double-float arithmetic (about 48 significant bits).  The chosen index is
// therefore the exact nearest code of the fp32 residual (lowest index on
// exact ties) unless two distances agree to ~13 significant digits.  The
// residual update is fp32.
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
constexpr int kNSlot = 2;                       // residual operand slots (groups in flight)
constexpr int kCbStages = 2;                    // codebook ring
constexpr uint32_t kBlockBytes = kTile * 128;   // 128 rows x 64 bf16, 128B swizzled
constexpr uint32_t kFull = 0xffffffffu;
static_assert(kTile == 4 * 32, "one four-row gather per lane of the producer warp");

struct Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t zfull[2];
  uint64_t zempty[2];
  uint64_t uready[kNSlot];
  uint64_t dfull[2];
  uint64_t dempty[2];
  uint64_t pair[4];                 // the two epilogue warps of a TMEM quadrant
  uint64_t cbfull[kCbStages];       // codebook ring
  uint64_t cbempty[kCbStages];
  uint32_t tmem_base;
  int abort;
  float xb1[2][2][kTile];           // [item parity][half][row] best of a half
  float xb2[2][2][kTile];           // second best of a half
  int xk1[2][2][kTile];             // index of the best
  float nu[kNSlot][2][kTile];       // ||u|| of the residual in a slot [use parity]
  float uscr[8][32];                // per epilogue warp: the residual being refined
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

__device__ __forceinline__ void give_up(Ctl* ctl, int* err) {
  ctl->abort = 1;
  atomicOr(err, kErrTimeout);
}

struct Geo {
  int r, nkx, nkr, na, nP, nV, nh, nrow, GD, B, nzb, zstride, nsplit;
  bool share;   // anchor rows gathered once per block for all -M splits
};

__device__ __forceinline__ Geo geometry(const CompressArgs& a, bool vq) {
  Geo g;
  g.r = a.r;
  g.nkx = a.d / 64;
  g.nkr = a.re / 64;
  g.nsplit = a.nsplit;
  g.na = a.nsplit * g.nkr;
  g.nP = g.nkx + (a.anchor ? g.na : 0);
  g.nV = vq ? a.G * a.R : 0;
  g.nh = a.r > 256 ? 2 : 1;
  g.nrow = a.r > 256 ? 256 : a.r;
  g.GD = a.gd;
  g.B = a.G < kNSlot ? a.G : kNSlot;
  g.nzb = vq ? (a.r <= 128 ? 2 : 1) : (2 * a.r <= 512 ? 2 : 1);
  g.zstride = a.r;
  g.share = a.nsplit > 1 && a.nstage >= a.nsplit;
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
// (four interleaved trackers; exact ties keep the lowest index).
__device__ __forceinline__ void scan_half(uint32_t tdist, const float* cn, int KH, int koff,
                                          float& b1, float& b2, int& k1) {
  const float inf = __int_as_float(0x7f800000);
  float t1[4] = {inf, inf, inf, inf}, t2[4] = {inf, inf, inf, inf};
  int tk[4] = {0, 0, 0, 0};
  for (int c0 = 0; c0 < KH; c0 += 32) {
    float v[32];
    tmem_ld32(tdist + c0, v);
    float cv[32];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 f = reinterpret_cast<const float4*>(cn + c0)[q];
      cv[4 * q] = f.x;
      cv[4 * q + 1] = f.y;
      cv[4 * q + 2] = f.z;
      cv[4 * q + 3] = f.w;
    }
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float D = fmaf(-2.f, v[j + u], cv[j + u]);
        t2[u] = fminf(t2[u], fmaxf(t1[u], D));
        tk[u] = D < t1[u] ? (koff + c0 + j + u) : tk[u];
        t1[u] = fminf(t1[u], D);
      }
    }
  }
  b1 = t1[0];
  k1 = tk[0];
  b2 = t2[0];
#pragma unroll
  for (int u = 1; u < 4; ++u) {
    b2 = fminf(fminf(b2, t2[u]), fmaxf(b1, t1[u]));
    if (t1[u] < b1 || (t1[u] == b1 && tk[u] < k1)) {
      b1 = t1[u];
      k1 = tk[u];
    }
  }
}

// a + b = s + e exactly (Knuth's two-sum)
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// 16-byte chunk c of code k in a codebook stage as TMA wrote it (rows of
// 2*GD bytes, 64- or 32-byte swizzle: the chunk index is XORed with address
// bits 7.. of the row).
template <int GD>
__device__ __forceinline__ uint4 code_chunk(const uint8_t* stage, int k, int c) {
  constexpr int kRowB = 2 * GD, kNch = kRowB / 16;
  const int sw = c ^ (((k * kRowB) >> 7) & (kNch - 1));
  return *reinterpret_cast<const uint4*>(stage + k * kRowB + sw * 16);
}

// Element `lane` (< GD) of code k in a codebook stage, as a float.
template <int GD>
__device__ __forceinline__ float code_elem(const uint8_t* stage, int k, int lane) {
  constexpr int kRowB = 2 * GD, kNch = kRowB / 16;
  const int c = lane >> 3;
  const int sw = c ^ (((k * kRowB) >> 7) & (kNch - 1));
  const __nv_bfloat16 v =
      *reinterpret_cast<const __nv_bfloat16*>(stage + k * kRowB + sw * 16 + (lane & 7) * 2);
  return __bfloat162float(v);
}

// ||u - c_k||^2 as an unevaluated pair hi + lo (about 48 significant bits),
// computed by the whole warp: lane j forms (u_j - c_j)^2 exactly (two-sum of
// the difference, fma split of the square) and a five-level shuffle tree
// adds the 32 pairs with two-sums.  `uj` is u_j on lane j (0 past GD).
// Enough to order two codes whose distances differ in the 13th digit.
template <int GD>
__device__ __forceinline__ void coop_exact_dist(float uj, const uint8_t* stage, int k, int lane,
                                                float& hi, float& lo) {
  float h = 0.f, l = 0.f;
  if (lane < GD) {
    float d, de;
    two_sum(uj, -code_elem<GD>(stage, k, lane), d, de);
    h = d * d;
    l = fmaf(2.f * d, de, fmaf(d, d, -h));
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float oh = __shfl_xor_sync(kFull, h, o);
    const float ol = __shfl_xor_sync(kFull, l, o);
    float s, e;
    two_sum(h, oh, s, e);
    h = s;
    l = (l + ol) + e;
  }
  two_sum(h, l, hi, lo);
}

// Rare path, on CUDA cores (the distance buffer is already released): for
// every lane with `need`, the warp recomputes coarse distances
// ||c_k||^2 - 2 u.c_k in fp32 for all K codes from the codebook stage (lane j
// takes codes j, j + 32, ...), keeps the codes within that lane's `thr`, and
// re-scores each of them exactly with the whole warp.  Returns the exact
// nearest code (lowest index on exact ties); other lanes keep k_init.
template <int GD>
__device__ __forceinline__ int refine(const float (&u)[GD], const float* cn,
                                      const uint8_t* stage, float* uscr, int K, float thr,
                                      bool need, int k_init, int lane) {
  float bh = __int_as_float(0x7f800000), bl = 0.f;
  int kb = k_init;
  uint32_t lanes = __ballot_sync(kFull, need);
  while (lanes) {
    const int L = __ffs(lanes) - 1;
    lanes &= lanes - 1;
    __syncwarp();
    if (lane == L) {
#pragma unroll
      for (int i = 0; i < GD; ++i) uscr[i] = u[i];
    }
    __syncwarp();
    const float thrL = __shfl_sync(kFull, thr, L);
    float uu[GD];
#pragma unroll
    for (int i = 0; i < GD; ++i) uu[i] = uscr[i];
    uint32_t cmask = 0;   // bit i: code lane + 32 i is a candidate
#pragma unroll 1
    for (int i = 0; i < K / 32; ++i) {
      const int k = lane + 32 * i;
      float dot = 0.f;
#pragma unroll
      for (int q = 0; q < GD / 8; ++q) {
        const uint4 w = code_chunk<GD>(stage, k, q);
        const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(hp[e]);
          dot = fmaf(uu[q * 8 + 2 * e], f.x, dot);
          dot = fmaf(uu[q * 8 + 2 * e + 1], f.y, dot);
        }
      }
      cmask |= (fmaf(-2.f, dot, cn[k]) <= thrL ? 1u : 0u) << i;
    }
    const float uj = lane < GD ? uscr[lane] : 0.f;
#pragma unroll 1
    for (int i = 0; i < K / 32; ++i) {
      uint32_t cl = __ballot_sync(kFull, (cmask >> i) & 1u);
      while (cl) {
        const int kk = 32 * i + __ffs(cl) - 1;
        cl &= cl - 1;
        float eh, el;
        coop_exact_dist<GD>(uj, stage, kk, lane, eh, el);
        if (lane == L && (eh < bh || (eh == bh && el < bl))) {
          bh = eh;
          bl = el;
          kb = kk;
        }
      }
    }
  }
  return kb;
}

template <int GD>
__device__ void epilogue_vq(const CompressArgs& a, const Geo& geo, Ctl* ctl, uint32_t tbase,
                            uint32_t ubase, const float* cn_s, const uint8_t* cbring_p,
                            uint32_t cbsb, int tile, int zb, int q, int h, int lane,
                            uint32_t& dcnt, uint32_t& pcnt, uint32_t (&suse)[kNSlot],
                            bool& alive) {
  const int row = q * 32 + lane;
  const int n = tile * kTile + row;
  const bool store = n < a.N;
  bool bad = false;
  if (store && a.anchor) {
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
    // The residual of the group this warp owns in the batch (at most one:
    // batches start at even groups and hold two) lives in registers through
    // the rounds; Z's TMEM columns are only read here.
    float u[GD];
    // round-0 operands of the groups this half owns
    for (int g = b0; g < b1g; ++g) {
      if ((g & 1) != h && G > 1) continue;
      if (G == 1 && h == 1) continue;
      tmem_load_group<GD>(tz + g * GD, u);
      const int slot = g - b0;
      const float nu = write_operand<GD>(ubase + slot * kBlockBytes, row, u);
      // ||u|| slots alternate with the slot's uses, so a writer never
      // touches the one its partner warp may still be reading
      ctl->nu[slot][suse[slot] & 1u][row] = nu;
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
        const uint32_t npar = suse[slot] & 1u;   // parity of this use of the slot
        ++suse[slot];
        // this step's codebook stage (read by the owner's refinement and
        // residual update; the owners release it at the end of the step)
        const int cs = static_cast<int>(dcnt % kCbStages);
        const uint32_t cph = (dcnt / kCbStages) & 1u;
        const uint8_t* stage = cbring_p + cs * cbsb;
        // 1. distances of this half are in TMEM
        if (!warp_wait(smem_u32(&ctl->dfull[h]), dcnt & 1u, ctl, bud)) {
          give_up(ctl, a.err);
          alive = false;
          break;
        }
        tc_fence_after();
        if (owner && !warp_wait(smem_u32(&ctl->cbfull[cs]), cph, ctl, bud)) {
          give_up(ctl, a.err);
          alive = false;
          break;
        }
        const uint32_t tdist = tbase + lanebase + 256 + h * KH;
        float b1, b2;
        int k1;
        scan_half(tdist, cn_s + book * K + h * KH, KH, h * KH, b1, b2, k1);
        // release this half of the distance buffer at once: the next step's
        // MMA overlaps the merge and the update below (the rare refinement
        // recomputes what it needs on CUDA cores)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->dempty[h]));
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
        const float nu = ctl->nu[slot][npar][row];
        const float cm = __ldg(a.cmax + book);
        // certified bound on |D~_k - D_k| (two-term split, fp32 accumulation
        // of 2*GD exact products, fp32 rounding of ||c||^2 and the fma)
        const float eps = 2e-5f * nu * cm + 1.2e-7f * (cm * cm + 2.f * nu * cm + fabsf(B1));
        const bool need = (B2 - B1) <= 2.f * eps;
        if (owner && __any_sync(kFull, need)) {
          {
            // band of the candidates: the MMA-coarse band plus the error of
            // the fp32 CUDA-core dot products (32 exact products, fp32 sums)
            const float thr =
                B1 + 2.f * eps + 4e-6f * nu * cm + 2.4e-7f * (cm * cm + fabsf(B1));
            const int kb = refine<GD>(u, cn_s + book * K, stage, ctl->uscr[q + 4 * h], K, thr,
                                      need, K1, lane);
            if (need) K1 = kb;
          }
        }
        ++dcnt;
        if (!owner) continue;
        // 4. owner: record the index, update the residual, next operand
        if (store) idx_out[rho * G + g] = bad ? static_cast<uint8_t>(0) : static_cast<uint8_t>(K1);
        if (rho + 1 < R) {
#pragma unroll
          for (int c = 0; c < GD / 8; ++c) {
            const uint4 w = code_chunk<GD>(stage, K1, c);
            const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(hp[e]);
              u[c * 8 + 2 * e] -= f.x;
              u[c * 8 + 2 * e + 1] -= f.y;
            }
          }
          const float nn = write_operand<GD>(ubase + slot * kBlockBytes, row, u);
          ctl->nu[slot][suse[slot] & 1u][row] = nn;
          fence_async_shared();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctl->uready[slot]));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->cbempty[cs]));
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
  const uint32_t cbsb = vq ? static_cast<uint32_t>(a.K * a.gd) * 2u : 0u;   // codebook stage
  // shared memory: main ring | codebook ring | residual slots | ||c||^2 | ids | control
  const uint32_t ring = smem_u32(base);
  uint32_t off = nst * sb;
  const uint32_t cbring = ring + off;
  off += kCbStages * cbsb;
  const uint32_t ubase = ring + off;
  off += vq ? geo.B * kBlockBytes : 0u;
  float* cn_s = reinterpret_cast<float*>(base + off);
  off += vq ? ((static_cast<uint32_t>(a.R * a.G * a.K) * 4u + 15u) & ~15u) : 0u;
  int* tids_s = reinterpret_cast<int*>(base + off);   // [2][kTile], producer only
  off += 2 * kTile * 4;
  Ctl* ctl = reinterpret_cast<Ctl*>(base + off);

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
    for (int s = 0; s < kCbStages; ++s) {
      mbar_init(smem_u32(&ctl->cbfull[s]), 1);
      mbar_init(smem_u32(&ctl->cbempty[s]), 4);   // the four owner warps of the step
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
  const uint64_t bud = a.timeout_ns;

  if (warp == 0) {
    // --------------------------------------------- producer of the main ring
    // Lane 0 issues the TMA loads.  The whole warp stages each tile's anchor
    // row ids in shared memory, one tile ahead (invalid ids and rows past N
    // read row 0; their outputs are zeroed by the epilogue).
    if (lane == 0) {
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmAt);
      prefetch_tmap(&tmMt);
      prefetch_tmap(&tmE);
    }
    constexpr int kIdsPerLane = kTile / 32;
    auto fetch_ids = [&](int tile, int (&v)[kIdsPerLane]) {
#pragma unroll
      for (int j = 0; j < kIdsPerLane; ++j) {
        const int n = tile * kTile + lane + 32 * j;
        const int t = (a.anchor && n < a.N) ? __ldg(a.tids + n) : 0;
        v[j] = (t < 0 || t >= a.V) ? 0 : t;
      }
    };
    auto store_ids = [&](int buf, const int (&v)[kIdsPerLane]) {
#pragma unroll
      for (int j = 0; j < kIdsPerLane; ++j) tids_s[buf * kTile + lane + 32 * j] = v[j];
    };
    if (L > 0) {
      int v[kIdsPerLane];
      fetch_ids(blockIdx.x, v);
      store_ids(0, v);
    }
    __syncwarp();
    int s = 0;
    uint32_t ph = 0;   // phase parity of stage s
    bool ok = true;
    for (int it = 0; it < L && ok; ++it) {
      const int tile = blockIdx.x + it * gridDim.x;
      int nv[kIdsPerLane];
      if (it + 1 < L) fetch_ids(tile + gridDim.x, nv);
      {
        // the whole warp walks the items: lane 0 issues the block loads,
        // every lane one of the 32 four-row gathers of an anchor block (a
        // single thread issuing them all would hold the tile back)
        const int* ts = tids_s + (it & 1) * kTile;
        for (int p = 0; p < geo.nP; ++p) {
          if (!(ok = warp_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, ctl, bud))) break;
          const uint32_t st = ring + s * sb;
          const uint32_t fb = smem_u32(&ctl->full[s]);
          if (p < geo.nkx) {
            if (lane == 0) {
              mbar_arrive_expect_tx(fb, kBlockBytes + geo.r * 128u);
              tma_load_2d(st, &tmX, p * 64, tile * kTile, fb);
              for (int hh = 0; hh < geo.nh; ++hh)
                tma_load_2d(st + kBlockBytes + hh * 256u * 128u, &tmAt, p * 64, hh * 256, fb);
            }
          } else {
            // anchor item (kb, sp): -M^T split sp, block kb; the anchor rows
            // E[tids] of block kb come with sp == 0 (or every sp when the
            // ring is too short to keep that stage while the other splits
            // stream)
            const int j = p - geo.nkx, kb = j / geo.nsplit, sp = j - kb * geo.nsplit;
            const bool gather = sp == 0 || !geo.share;
            if (lane == 0) {
              mbar_arrive_expect_tx(fb, (gather ? kBlockBytes : 0u) + geo.r * 128u);
              for (int hh = 0; hh < geo.nh; ++hh)
                tma_load_2d(st + kBlockBytes + hh * 256u * 128u, &tmMt, kb * 64,
                            sp * geo.r + hh * geo.nrow, fb);
            }
            // full[s] completes only when every byte armed above has landed,
            // so the lanes' gathers may be issued in any order around it
            if (gather)
              tma_gather4(st + lane * 512, &tmE, kb * 64, ts[4 * lane], ts[4 * lane + 1],
                          ts[4 * lane + 2], ts[4 * lane + 3], fb);
          }
          if (++s == nst) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // the gathers that read this buffer two tiles ago were issued already
      // (their row ids travel with the instruction)
      if (it + 1 < L) store_ids((it + 1) & 1, nv);
      __syncwarp();
    }
    if (!ok && lane == 0) give_up(ctl, a.err);
  } else if (warp == 2 && lane == 0 && vq) {
    // ------------------------------------------ producer of the codebook ring
    prefetch_tmap(&tmC);
    int c = 0;
    bool ok = true;
    for (int it = 0; it < L && ok; ++it)
      for (int b0 = 0; b0 < a.G && ok; b0 += geo.B) {
        const int b1g = b0 + geo.B < a.G ? b0 + geo.B : a.G;
        for (int rho = 0; rho < a.R && ok; ++rho)
          for (int g = b0; g < b1g && ok; ++g, ++c) {
            const int s = c % kCbStages, use = c / kCbStages;
            if (!(ok = mbar_wait(smem_u32(&ctl->cbempty[s]), (use & 1) ^ 1, &ctl->abort, bud)))
              break;
            const uint32_t fb = smem_u32(&ctl->cbfull[s]);
            mbar_arrive_expect_tx(fb, cbsb);
            tma_load_2d(cbring + s * cbsb, &tmC, 0, (rho * a.G + g) * a.K, fb);
          }
      }
    if (!ok) give_up(ctl, a.err);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    // One thread issues every tcgen05 operation of the CTA.  It interleaves
    // two independent streams with non-blocking probes: the VQ distance MMAs
    // of the tile in the epilogue (first, they gate the epilogue) and the
    // projection MMAs of the next tile.  Each stream consumes its own ring in
    // order, so no probe can see a phase two behind.  The loop is kept lean
    // (no divisions, descriptors advanced by offsets): this thread shares its
    // scheduler with two busy epilogue warps.
    const uint32_t idz = idesc_bf16(kTile, geo.nrow);
    const uint32_t idd = idesc_bf16(kTile, vq ? a.K : 16);
    // distance MMA: K-steps over [u_hi | u_lo]; both halves read the same
    // code rows (one copy of each code in the codebook ring)
    constexpr int kStepsC = (GD > 0 ? GD : 16) / 16;
    const uint64_t ring_d = sw128_desc(ring);
    const uint64_t ub_d = sw128_desc(ubase);
    const uint64_t cb_d = narrow_desc<(GD == 32 ? 64 : 32)>(cbring);
    int pj_it = 0, pj_p = 0, pj_s = 0, pj_sp = 0, blk0 = 0, blk1 = 0;
    uint32_t pj_ph = 0;
    bool pj_started = false;
    int vq_it = 0, vq_b0 = 0, vq_rho = 0, vq_g = 0, vq_cs = 0;
    uint32_t vq_cph = 0, e = 0;
    uint32_t ucnt0 = 0, ucnt1 = 0;
    bool got_u = false, got_c = false;
    const int vq_end = vq ? L : 0;
    uint64_t last = global_ns();
    uint32_t idle = 0;
    bool ok = true;
    while (ok && (pj_it < L || vq_it < vq_end)) {
      bool progressed = false;
      if (vq_it < vq_end) {
        const int slot = vq_g - vq_b0;
        if (!got_u)
          got_u = mbar_test(smem_u32(&ctl->uready[slot]), (slot == 0 ? ucnt0 : ucnt1) & 1u);
        if (!got_c) got_c = mbar_test(smem_u32(&ctl->cbfull[vq_cs]), vq_cph);
        if (got_u && got_c && mbar_test(smem_u32(&ctl->dempty[0]), (e & 1u) ^ 1u) &&
            mbar_test(smem_u32(&ctl->dempty[1]), (e & 1u) ^ 1u)) {
          // one MMA over all K codes: both halves of the distance buffer
          tc_fence_after();
          const uint64_t ad = ub_d + ((static_cast<uint32_t>(slot) * kBlockBytes) >> 4);
          const uint64_t bd = cb_d + ((static_cast<uint32_t>(vq_cs) * cbsb) >> 4);
#pragma unroll
          for (int k = 0; k < 2 * kStepsC; ++k)
            mma_bf16(tbase + 256, ad + 2 * k, bd + 2 * (k % kStepsC), idd, k != 0 ? 1u : 0u);
          mma_commit(smem_u32(&ctl->dfull[0]));
          mma_commit(smem_u32(&ctl->dfull[1]));
          progressed = true;
          if (slot == 0) ++ucnt0; else ++ucnt1;
          got_u = got_c = false;
          ++e;
          if (++vq_cs == kCbStages) {
            vq_cs = 0;
            vq_cph ^= 1u;
          }
          const int b1g = vq_b0 + geo.B < a.G ? vq_b0 + geo.B : a.G;
          if (++vq_g == b1g) {
            vq_g = vq_b0;
            if (++vq_rho == a.R) {
              vq_rho = 0;
              vq_b0 += geo.B;
              vq_g = vq_b0;
              if (vq_b0 >= a.G) {
                vq_b0 = vq_g = 0;
                ++vq_it;
              }
            }
          }
        }
      }
      // projection MMAs only while the VQ stream waits: the tensor pipe runs
      // in order, so a projection item queued ahead of a distance MMA would
      // delay the epilogue, which is the critical path
      if (pj_it < L && !progressed) {
        const int zb = geo.nzb == 2 ? (pj_it & 1) : 0;
        const int zuse = geo.nzb == 2 ? (pj_it >> 1) : pj_it;
        if (!pj_started && mbar_test(smem_u32(&ctl->zempty[zb]), (zuse & 1) ^ 1)) {
          pj_started = true;
          tc_fence_after();
        }
        if (pj_started && mbar_test(smem_u32(&ctl->full[pj_s]), pj_ph)) {
          tc_fence_after();
          const uint32_t dz = tbase + zb * geo.zstride;
          const bool anchor = pj_p >= geo.nkx;
          if (anchor && pj_sp == 0) blk0 = pj_s;
          if (anchor && pj_sp == 1) blk1 = pj_s;
          // A operand: this stage, or for a shared anchor split the stage of
          // split 0 of the same block (still held)
          const int sa_s = (anchor && geo.share && pj_sp > 0) ? blk0 : pj_s;
          const uint64_t ad = ring_d + ((static_cast<uint32_t>(sa_s) * sb) >> 4);
          const uint64_t bd = ring_d + ((static_cast<uint32_t>(pj_s) * sb + kBlockBytes) >> 4);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            for (int hh = 0; hh < geo.nh; ++hh)
              mma_bf16(dz + hh * 256, ad + 2 * k, bd + hh * ((256u * 128u) >> 4) + 2 * k, idz,
                       (pj_p | k) != 0 ? 1u : 0u);
          if (!anchor || !geo.share) {
            mma_commit(smem_u32(&ctl->empty[pj_s]));
          } else if (pj_sp == geo.nsplit - 1) {
            // release the block's stages together (split 0 held the rows)
            mma_commit(smem_u32(&ctl->empty[blk0]));
            if (geo.nsplit > 2) mma_commit(smem_u32(&ctl->empty[blk1]));
            mma_commit(smem_u32(&ctl->empty[pj_s]));
          }
          progressed = true;
          if (++pj_s == nst) {
            pj_s = 0;
            pj_ph ^= 1u;
          }
          if (anchor && ++pj_sp == geo.nsplit) pj_sp = 0;
          if (++pj_p == geo.nP) {
            mma_commit(smem_u32(&ctl->zfull[zb]));
            pj_p = 0;
            pj_sp = 0;
            pj_started = false;
            ++pj_it;
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
    if (vq) {
      const int ncn = a.R * a.G * a.K;
      for (int x = threadIdx.x - kEpiWarp0 * 32; x < ncn; x += 8 * 32) cn_s[x] = __ldg(a.cnorm + x);
      named_bar_sync(1, 8 * 32);
    }
    uint32_t dcnt = 0, pcnt = 0;
    uint32_t suse[kNSlot] = {0u, 0u};   // uses of each residual slot so far
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
          epilogue_vq<GD>(a, geo, ctl, tbase, ubase, cn_s, base + nst * sb, cbsb, tile, zb, q,
                          h, lane, dcnt, pcnt, suse, alive);
        const int n = tile * kTile + q * 32 + lane;
        if (alive && h == 0 && n < a.N && a.anchor) {   // no token ids without the anchor
          const int t = a.tids[n];
          if (t < 0 || t >= a.V) atomicOr(a.err, kErrBadToken);
        }
      } else {
        const int row = q * 32 + lane;
        const int n = tile * kTile + row;
        const bool store = n < a.N;
        bool bad = false;
        if (store && a.anchor) {
          const int t = a.tids[n];
          bad = t < 0 || t >= a.V;
          if (bad && h == 0) atomicOr(a.err, kErrBadToken);
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
