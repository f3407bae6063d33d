// kernels_compress_pipe.cu -- pipelined persistent compress kernel (r <= 256
// without VQ, r <= 128 with VQ).
//
// MAPL §3.2 eq. (1) with the anchor folded through M = P_send A:
//     Z = X A - E_send[tids] M          (one TMEM accumulation per tile)
// and, with VQ, the multi-codebook residual quantisation of §3.5: for every
// group g and round rho the nearest code of the group's residual.
//
// Each CTA owns one contiguous range of about N / gridDim.x tokens and walks
// it in tiles of up to 128 rows (the MMA's M), so every SM streams the same
// number of X rows.  Warp roles (12 warps):
//   warp 0        : TMA producer of the X ring: the tile's X blocks (HBM),
//                   then the anchor rows E[tids] of each 64-column anchor
//                   block (tile::gather4, one four-row gather per lane).
//   warp 3 lane 0 : TMA producer of the B ring: A^T blocks, then the -M^T
//                   split blocks.  A^T comes from L2, so this ring is kept
//                   shallow and the X ring deep: the two advance on their own.
//   warp 2 lane 0 : TMA producer of the codebook ring (one book per VQ step)
//                   and issuer of the VQ distance products, in 128-code
//                   chunks, of two independent step streams (one per
//                   epilogue warp set).
//   warp 1        : TMEM allocation; lane 0 issues the projection of each
//                   tile into the Z accumulator.
//   warps 4..11   : epilogue.  Warp w reads TMEM lanes 32 (w % 4).. (its token
//                   rows); warp set j = (w - 4) / 4 owns the groups g = j mod 2
//                   of those rows: their residuals stay in its registers through
//                   all rounds, it scans every code of its own steps, so no
//                   result is merged across warps.
//
// VQ step (group g, round rho) of a warp set.  The residual u (fp32) is split
// into u_hi = bf16(u) and u_lo = bf16(u - u_hi), and -u_hi, -u_lo are written
// to a TMEM operand slot (two per set, alternating between consecutive steps,
// so the next step's operand is in place while this one is scanned).  One
// accumulation per 128-code chunk gives
//     t_k = ||c_k||^2 / 2 - u_hi.c_k - u_lo.c_k  (= D~_k / 2),
// the norm entering as one more K = 16 product of a constant shared-memory
// tile of rows [1, 1, 1, 0, ...] with the book's rows [h_hi, h_mid, h_lo, 0,
// ...], the three bf16 terms of the fp32 ||c_k||^2 / 2 (loaded with the
// codes), so the scan reads the distances straight from TMEM.  The chunk
// lands in one TMEM slot per set; the other set's chunk is computed while
// this one is scanned, and the slot is released as soon as its last quarter
// is loaded.  Each 32-code quarter is scanned in two passes: its minimum
// (three-input minimums), then on the FMA pipe a saturated indicator of every
// code within a certified band of the running minimum, summed with weights
// 1 + k / 1024 so that the count of such codes and, when it is one, the
// code's index are both exact in fp32.  The band bounds the error of the
// split, of the norm's split and of the fp32 accumulation, so when one code
// is inside it that code is the exact nearest code of the fp32 residual;
// otherwise (rare) every code of the 32-code quarters that held a candidate
// is re-scored on CUDA cores with a double-float squared distance, lowest
// index on exact ties.  The residual update is fp32.
//
// Every wait is time bounded (mbar_wait); a CTA that gives up sets the device
// error word, waits (bounded) for its own copies and products in flight, and
// leaves through the common exit that frees TMEM.
#include "mapl_internal.h"
#include "pdl.cuh"
#include "ptx.cuh"

namespace mapl {

namespace {

constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kMaxX = 12;
constexpr int kMaxB = 8;
constexpr int kMaxC = 4;
constexpr uint32_t kXBytes = kTile * 128;   // 128 rows x 64 bf16, 128B swizzled
constexpr uint32_t kFull = 0xffffffffu;
constexpr uint32_t kColOp = 128;            // TMEM columns of the operand slots
constexpr uint32_t kColDist = 256;          // TMEM columns of the distance chunk slots
constexpr int kChunk = 128;                 // codes per distance MMA (one TMEM slot per set)
constexpr uint32_t kOnesBytes = 128 * 32;   // A tile of the norm product: 128 rows x 16 bf16
static_assert(kTile == 4 * 32, "one four-row gather per lane of the producer warp");

struct Ctl {
  uint64_t xfull[kMaxX], xempty[kMaxX];
  uint64_t bfull[kMaxB], bempty[kMaxB];
  uint64_t cfull[kMaxC], cempty[kMaxC];
  uint64_t zfull[2], zempty[2];
  uint64_t opready[4];              // [set][slot]
  uint64_t dfull[2], dempty[2];     // per warp set: its distance chunk slot
  uint64_t mmadone;                 // projection issuer's last products
  uint64_t vqdone;                  // distance-product issuer's last products
  uint32_t tmem_base;
  int abort;
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

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, Ctl* ctl,
                                          uint64_t budget) {
  const bool ok = mbar_wait_sleep(bar, parity, &ctl->abort, budget);
  return __all_sync(kFull, ok);
}

// Bounded wait that ignores the abort flag: used on the way out, to let this
// thread's own copies or products finish before the CTA frees its memory.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t budget) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > budget) return;
}

constexpr uint64_t kDrainNs = 10000000ull;   // 10 ms

// Rows [t0, t0 + cnt) of tile `it` of this CTA's contiguous token range.
struct Range {
  int row0, row1, ntile;
  __device__ __forceinline__ int t0(int it) const { return row0 + it * kTile; }
  __device__ __forceinline__ int cnt(int it) const {
    const int c = row1 - t0(it);
    return c < kTile ? c : kTile;
  }
};

__device__ __forceinline__ Range cta_range(int N) {
  Range r;
  r.row0 = static_cast<int>(static_cast<long long>(N) * blockIdx.x / gridDim.x);
  r.row1 = static_cast<int>(static_cast<long long>(N) * (blockIdx.x + 1) / gridDim.x);
  r.ntile = (r.row1 - r.row0 + kTile - 1) / kTile;
  return r;
}

// Split of the negated residual into the TMEM operand [-u_hi (GD) | -u_lo
// (GD)] of the distance MMA, two bf16 per column (negation is exact and
// commutes with round-to-nearest, so these are the negated terms of u's own
// split); returns ||u|| rounded up.
template <int GD>
__device__ __forceinline__ float write_operand(uint32_t taddr, const float (&u)[GD]) {
  uint32_t w[GD];
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < GD / 2; ++e) {
    const float x0 = u[2 * e], x1 = u[2 * e + 1];
    s = fmaf(x0, x0, s);
    s = fmaf(x1, x1, s);
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    w[e] = *reinterpret_cast<const uint32_t*>(&h) ^ 0x80008000u;
    w[GD / 2 + e] = *reinterpret_cast<const uint32_t*>(&l) ^ 0x80008000u;
  }
  if constexpr (GD == 32)
    tmem_st32u(taddr, w);
  else
    tmem_st16u(taddr, w);
  tmem_wait_st();
  return sqrtf(s) * 1.000001f;
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
// the difference, fma split of the square) and a five-level shuffle tree adds
// the 32 pairs with two-sums.  `uj` is u_j on lane j (0 past GD).
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

// Rare path on CUDA cores: the exact nearest code for every lane with
// `need`.  A lane's candidates lie in the 32-code halves of its `halves`
// mask (bit h: codes 32 h .. 32 h + 31 had a code within the band when they
// were scanned).  For each such half the warp recomputes the coarse distance
// ||c_k||^2 - 2 u.c_k of its 32 codes in fp32 (one code per lane), keeps
// those within `thr`, and re-scores each with the double-float squared
// distance of coop_exact_dist.  Returns the exact nearest code (lowest index
// on exact ties); other lanes keep k_init.
template <int GD>
__device__ __forceinline__ int refine(const float (&u)[GD], const float* cn, const uint8_t* stage,
                                      float* uscr, float thr, uint32_t halves, bool need,
                                      int k_init, int lane) {
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
    uint32_t hm = __shfl_sync(kFull, halves, L);
    const float uj = lane < GD ? uscr[lane] : 0.f;
    while (hm) {
      const int h = __ffs(hm) - 1;
      hm &= hm - 1;
      const int k = 32 * h + lane;
      float dot = 0.f;
#pragma unroll
      for (int qq = 0; qq < GD / 8; ++qq) {
        const uint4 w = code_chunk<GD>(stage, k, qq);
        const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(hp[e]);
          dot = fmaf(uscr[qq * 8 + 2 * e], f.x, dot);
          dot = fmaf(uscr[qq * 8 + 2 * e + 1], f.y, dot);
        }
      }
      uint32_t cl = __ballot_sync(kFull, fmaf(-2.f, dot, __ldg(cn + k)) <= thrL);
      while (cl) {
        const int kk = 32 * h + __ffs(cl) - 1;
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

// min(max(a * b + c, 0), 1) in one FMA-pipe instruction.
__device__ __forceinline__ float fma_sat(float a, float b, float c) {
  float r;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// A quarter of a 128-code chunk of the distance scan (32 codes), two passes over
// the registers, which hold t_k = ||c_k||^2 / 2 - u.c_k = D~_k / 2 as the
// distance MMA left it.  Pass 1: the minimum m (three-input minimums, the
// only ALU-pipe work).  Pass 2, on the FMA pipe: with thr = min(T, m) + band
// (T the minimum of the step's earlier codes), sat((thr - t_k) 2^60) is 1
// for every code below thr and 0 for every code at or above it, and acc =
// sum of sat(...) (1 + k / 1024) holds the number of those codes in its
// integer part and, when there is exactly one, its index k (< 32) in the
// fraction, both exact in fp32.  Returns m.
__device__ __forceinline__ float scan_half(const float (&v)[32], float T, float band, float& acc) {
  float t[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) t[i] = fmin3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  t[10] = fminf(v[30], v[31]);
  const float m = fminf(fmin3(fmin3(t[0], t[1], t[2]), fmin3(t[3], t[4], t[5]),
                              fmin3(t[6], t[7], t[8])),
                        fminf(t[9], t[10]));
  const float big = 0x1p60f;
  const float tb = (fminf(T, m) + band) * big;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    a0 = fmaf(fma_sat(v[i], -big, tb), 1.f + i * (1.f / 1024.f), a0);
    a1 = fmaf(fma_sat(v[i + 1], -big, tb), 1.f + (i + 1) * (1.f / 1024.f), a1);
    a2 = fmaf(fma_sat(v[i + 2], -big, tb), 1.f + (i + 2) * (1.f / 1024.f), a2);
    a3 = fmaf(fma_sat(v[i + 3], -big, tb), 1.f + (i + 3) * (1.f / 1024.f), a3);
  }
  acc = (a0 + a1) + (a2 + a3);
  return m;
}

// Merge one scanned half (codes base..base+31) into the step state: minimum
// T, an upper bound n on the codes within `band` of T (2 stands for "two or
// more"), when n == 1 that code's index k, and the mask of halves that held
// a code within the band when scanned (every code within the band of the
// final minimum is in one of them, since T only decreases).
__device__ __forceinline__ void merge_half(float m, float acc, int base, float band, float& T,
                                           int& n, int& k, uint32_t& halves) {
  if (acc >= 1.f) halves |= 1u << (base >> 5);
  // acc = count + index / 1024 for a single code; anything else (two or
  // more codes, a fraction from a distance within 2^-60 of the threshold)
  // counts as two
  int cnt = 0, first = 0;
  if (acc >= 1.f) {
    const float f = (acc - 1.f) * 1024.f;
    if (acc < 2.f && f == floorf(f) && f < 32.f) {
      cnt = 1;
      first = static_cast<int>(f);
    } else {
      cnt = 2;
    }
  }
  if (m < T - band) {
    // every earlier code is now outside the band
    n = cnt;
    k = base + first;
  } else if (m <= T + band) {
    n += cnt;
    if (m < T) k = base + first;
  }
  T = fminf(T, m);
}

// Per-CTA shared-memory layout (all ring stages 1024-byte aligned).
struct Smem {
  uint32_t xring, bring, cring, cn, ctl;
};

template <int GD, int NGW>
__device__ void epilogue_vq(const CompressArgs& a, Ctl* ctl, const Range& rg, uint32_t tbase,
                            const uint8_t* cring_p, uint32_t cbsb, int q, int j, int lane) {
  const int G = a.G, R = a.R, K = a.K, RG = a.R * a.G;
  const int nch = K / kChunk;
  const int nstep = R * NGW;   // steps of this set per tile
  const uint64_t bud = a.timeout_ns;
  const uint32_t lanebase = static_cast<uint32_t>(q * 32) << 16;
  const uint32_t top = tbase + lanebase + kColOp;
  const uint32_t tdist = tbase + lanebase + kColDist;
  float* uscr = ctl->uscr[q + 4 * j];
  uint32_t zcnt = 0;      // uses of the Z accumulator
  uint32_t gwrite = 0;    // operands written so far (all tiles); slot = gwrite & 1
  uint32_t cc = 0;        // distance chunks consumed so far
  uint32_t gstep = 0;     // steps completed so far (all tiles)
  bool alive = true;

  for (int it = 0; it < rg.ntile && alive; ++it) {
    const int t0 = rg.t0(it), tcnt = rg.cnt(it);
    const int row = q * 32 + lane;
    const int n = t0 + row;
    const bool valid = row < tcnt;
    bool bad = false;
    if (valid && a.anchor) {
      const int t = a.tids[n];
      bad = t < 0 || t >= a.V;
      if (bad && j == 0) atomicOr(a.err, kErrBadToken);
    }
    // residuals of this set's groups, loaded once from Z
    float u[NGW][GD];
    float nu[NGW];
    if (!warp_wait(smem_u32(&ctl->zfull[0]), zcnt & 1u, ctl, bud)) {
      give_up(ctl, a.err);
      break;
    }
    ++zcnt;
    tc_fence_after();
#pragma unroll
    for (int gi = 0; gi < NGW; ++gi) {
      const uint32_t col = static_cast<uint32_t>((2 * gi + j) * GD);
#pragma unroll
      for (int c = 0; c < GD; c += 16) {
        float t[16];
        tmem_ld16(tbase + lanebase + col + c, t);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) u[gi][c + i] = t[i];
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&ctl->zempty[0]));

    // operands of the first steps (step t of the tile is group t % NGW of
    // round t / NGW; with NGW == 1 step 1 depends on step 0)
    constexpr int kAhead = NGW >= 2 ? 2 : 1;
#pragma unroll
    for (int t = 0; t < kAhead; ++t) {
      const uint32_t slot = gwrite & 1u;
      nu[t] = write_operand<GD>(top + (2 * j + slot) * 32, u[t]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->opready[2 * j + slot]));
      ++gwrite;
    }

    uint8_t* idx_out = reinterpret_cast<uint8_t*>(a.out) + static_cast<size_t>(n) * RG;
    for (int rho = 0; rho < R && alive; ++rho) {
#pragma unroll
      for (int gi = 0; gi < NGW; ++gi) {
        if (!alive) break;
        const int s = rho * NGW + gi;
        const int g = 2 * gi + j;
        const int book = rho * G + g;
        const int cs = 2 * j + static_cast<int>(gstep & 1u);   // this set's book stage
        const uint32_t cph = (gstep >> 1) & 1u;
        const float* cn = a.cnorm + book * K;
        // band = twice the certified bound on |D~_k - D_k| for every code of
        // the book (the two-term split of u, |u - u_hi - u_lo| <= 2^-17 |u|;
        // fp32 accumulation of 2 GD + 3 exact products, ||c||^2 / 2 among
        // them; fp32 rounding of ||c||^2 and of its three-term split;
        // |D~| <= ||c||^2 + 2 ||u|| ||c||), widened for the rounding of the
        // scan's threshold test.  The scan runs on t = D~ / 2, so with half
        // the band.
        const float cm = __ldg(a.cmax + book);
        const float nuv = nu[gi];
        const float dmax = cm * cm + 2.f * nuv * cm;
        const float band = 2.f * (2e-5f * nuv * cm + 4.2e-6f * dmax) * 1.001f + 2.4e-7f * dmax;
        const float band_t = 0.5f * band;
        // 1. scan all chunks of this step, keeping the step minimum T (of
        // t), an upper bound n on the number of codes within `band_t` of it
        // and, for n == 1, that code's index
        float T = __int_as_float(0x7f800000);
        int ncand = 0;
        int K1 = 0;
        uint32_t halves = 0;
        for (int c = 0; c < nch; ++c) {
          const uint32_t ds = static_cast<uint32_t>(j);   // this set's chunk slot
          if (!warp_wait(smem_u32(&ctl->dfull[ds]), cc & 1u, ctl, bud)) {
            give_up(ctl, a.err);
            alive = false;
            break;
          }
          tc_fence_after();
          // the chunk in four quarters of 32 codes, each quarter's TMEM load
          // overlapping the previous quarter's scan; the slot is released
          // once the last quarter is in registers
          const uint32_t td = tdist + ds * kChunk;
          const int c0 = c * kChunk;
          float v[32], w[32];
          float acc;
          tmem_ld32(td, v);
          tmem_wait_ld();
          tmem_ld32(td + 32, w);
          float m = scan_half(v, T, band_t, acc);
          merge_half(m, acc, c0, band_t, T, ncand, K1, halves);
          tmem_wait_ld();
          tmem_ld32(td + 64, v);
          m = scan_half(w, T, band_t, acc);
          merge_half(m, acc, c0 + 32, band_t, T, ncand, K1, halves);
          tmem_wait_ld();
          tmem_ld32(td + 96, w);
          m = scan_half(v, T, band_t, acc);
          merge_half(m, acc, c0 + 64, band_t, T, ncand, K1, halves);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctl->dempty[ds]));
          ++cc;
          m = scan_half(w, T, band_t, acc);
          merge_half(m, acc, c0 + 96, band_t, T, ncand, K1, halves);
        }
        if (!alive) break;
        // 2. decision: a single code within the band of the minimum is the
        // exact nearest code; several (or none: non-finite distances) are
        // re-scored exactly
        const bool need = valid && ncand != 1;
        // the codebook stage is read below (refinement, residual update)
        if (!warp_wait(smem_u32(&ctl->cfull[cs]), cph, ctl, bud)) {
          give_up(ctl, a.err);
          alive = false;
          break;
        }
        const uint8_t* stage = cring_p + cs * cbsb;
        if (__any_sync(kFull, need)) {
          // band of the candidates, in D~: the MMA band plus the error of
          // the fp32 CUDA-core dot products (GD exact products, fp32 sums)
          const float thr = 2.f * T + band + 4e-6f * nuv * cm + 2.4e-7f * dmax;
          const int kb = refine<GD>(u[gi], cn, stage, uscr, thr, halves, need, K1, lane);
          if (need) K1 = kb;
        }
        // 3. index, residual update, next operand
        if (valid) idx_out[rho * G + g] = bad ? static_cast<uint8_t>(0) : static_cast<uint8_t>(K1);
        if (rho + 1 < R) {
#pragma unroll
          for (int c = 0; c < GD / 8; ++c) {
            const uint4 w = code_chunk<GD>(stage, K1, c);
            const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(hp[e]);
              u[gi][c * 8 + 2 * e] -= f.x;
              u[gi][c * 8 + 2 * e + 1] -= f.y;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->cempty[cs]));
        ++gstep;
        // operand of step s + kAhead (its group's residual is final now)
        if (s + kAhead < nstep) {
          const int gn = (gi + kAhead) % NGW;
          const uint32_t slot = gwrite & 1u;
          nu[gn] = write_operand<GD>(top + (2 * j + slot) * 32, u[gn]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctl->opready[2 * j + slot]));
          ++gwrite;
        }
      }
    }
  }
}

template <int GD, int NGW>
__global__ void __launch_bounds__(kThreads, 1)
    k_compress_pipe(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmAt,
                    const __grid_constant__ CUtensorMap tmMt, const __grid_constant__ CUtensorMap tmC,
                    const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmE,
                    const CompressArgs a) {
  // the next kernel in the stream may start its setup as this one's CTAs
  // leave; this kernel's own setup (barriers, TMEM, the constant tile)
  // overlaps the previous kernel, and nothing in memory is touched before
  // pdl_wait_prior below
  pdl_allow_next();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  constexpr bool vq = GD > 0;
  const int nx = a.nstage, nb = a.nbstage, ncb = vq ? a.ncb : 0;
  const uint32_t bsb = a.bstage_bytes;
  const uint32_t cbsb = a.cstage_bytes;
  // shared memory: X ring | B ring | codebook ring (two stages per warp set;
  // a stage holds the book's codes, then its rows [h_hi, h_mid, h_lo, 0...]
  // of ||c||^2 / 2 in three bf16 terms) | the constant A tile of the norm
  // product (VQ) | control
  const uint32_t xring = smem_u32(base);
  uint32_t off = nx * kXBytes;
  const uint32_t bring = xring + off;
  off += nb * bsb;
  const uint32_t cring = xring + off;
  const uint32_t cring_off = off;
  off += ncb * cbsb;
  const uint32_t ones = xring + off;
  if (vq) off += kOnesBytes;
  Ctl* ctl = reinterpret_cast<Ctl*>(base + off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Range rg = cta_range(a.N);
  const int L = rg.ntile;
  const int nkx = a.d / 64;
  const int neb = a.anchor ? a.re / 64 : 0;
  const int nsp = a.nsplit;
  const int nz = vq ? 1 : 2;                   // Z accumulators
  const uint32_t tmem_cols = vq ? 512u : (2u * a.r <= 32u ? 32u : (2u * a.r <= 64u ? 64u
                               : (2u * a.r <= 128u ? 128u : (2u * a.r <= 256u ? 256u : 512u))));

  if (threadIdx.x == 0) {
    for (int s = 0; s < nx; ++s) {
      mbar_init(smem_u32(&ctl->xfull[s]), 1);
      mbar_init(smem_u32(&ctl->xempty[s]), 1);
    }
    for (int s = 0; s < nb; ++s) {
      mbar_init(smem_u32(&ctl->bfull[s]), 1);
      mbar_init(smem_u32(&ctl->bempty[s]), 1);
    }
    for (int s = 0; s < ncb; ++s) {
      mbar_init(smem_u32(&ctl->cfull[s]), 1);
      mbar_init(smem_u32(&ctl->cempty[s]), 4);   // the four warps of the set using the book
    }
    for (int z = 0; z < 2; ++z) {
      mbar_init(smem_u32(&ctl->zfull[z]), 1);
      mbar_init(smem_u32(&ctl->zempty[z]), 8);
    }
    for (int s = 0; s < 4; ++s) mbar_init(smem_u32(&ctl->opready[s]), 4);
    for (int j = 0; j < 2; ++j) {
      mbar_init(smem_u32(&ctl->dfull[j]), 1);
      mbar_init(smem_u32(&ctl->dempty[j]), 4);
    }
    mbar_init(smem_u32(&ctl->mmadone), 1);
    mbar_init(smem_u32(&ctl->vqdone), 1);
    ctl->abort = 0;
    fence_mbar_init();
    fence_async_shared();
  }
  if (warp == 1) tmem_alloc(smem_u32(&ctl->tmem_base), tmem_cols);
  if (vq && warp >= kEpiWarp0) {
    // the A operand of the norm product: 128 rows [1, 1, 1, 0, ..., 0] of 16
    // bf16 (32 bytes, the 32-byte swizzle: 16-byte chunk c of row i sits at
    // chunk c ^ ((i >> 2) & 1)); one 16-byte chunk per epilogue thread
    const int x = threadIdx.x - kEpiWarp0 * 32;   // 0..255
    const int row = x >> 1, chunk = x & 1;
    const bool lead = (chunk ^ ((row >> 2) & 1)) == 0;
    const uint32_t dst = ones + static_cast<uint32_t>(row * 32 + chunk * 16);
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %3};" ::"r"(dst),
                 "r"(lead ? 0x3F803F80u : 0u), "r"(lead ? 0x00003F80u : 0u), "r"(0u)
                 : "memory");
    fence_async_shared();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ctl->tmem_base;
  const uint64_t bud = a.timeout_ns;
  // the inputs (and the plan's tables) may come from the kernel before
  pdl_wait_prior();

  if (warp == 0) {
    // ------------------------------------------------------ X ring producer
    if (lane == 0) {
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmE);
    }
    int s = 0;
    uint32_t ph = 0;
    uint32_t armed = 0;   // bit s: stage s was armed at least once
    uint32_t last_ph = 0; // bit s: parity of the last arming of stage s
    bool ok = true;
    for (int it = 0; it < L && ok; ++it) {
      const int t0 = rg.t0(it), tcnt = rg.cnt(it);
      // this lane's four anchor rows (rows past the tile or bad ids read row 0;
      // their outputs are zeroed or dropped by the epilogue)
      int ids[4] = {0, 0, 0, 0};
      if (neb > 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int rr = 4 * lane + k;
          const int t = rr < tcnt ? __ldg(a.tids + t0 + rr) : 0;
          ids[k] = (t < 0 || t >= a.V) ? 0 : t;
        }
      }
      for (int p = 0; p < nkx + neb; ++p) {
        if (!(ok = warp_wait(smem_u32(&ctl->xempty[s]), ph ^ 1u, ctl, bud))) break;
        const uint32_t st = xring + s * kXBytes;
        const uint32_t fb = smem_u32(&ctl->xfull[s]);
        if (lane == 0) mbar_arrive_expect_tx(fb, kXBytes);
        __syncwarp();
        if (p < nkx) {
          if (lane == 0) tma_load_2d(st, &tmX, p * 64, t0, fb);
        } else {
          tma_gather4(st + lane * 512, &tmE, (p - nkx) * 64, ids[0], ids[1], ids[2], ids[3], fb);
        }
        armed |= 1u << s;
        last_ph = (last_ph & ~(1u << s)) | (ph << s);
        if (++s == nx) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok) {
      if (lane == 0) give_up(ctl, a.err);
      // let this warp's copies land before the CTA can exit
      for (int k = 0; k < nx; ++k)
        if ((armed >> k) & 1u)
          drain_wait(smem_u32(&ctl->xfull[k]), (last_ph >> k) & 1u, kDrainNs);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------ B ring producer
    if (lane == 0) {
      prefetch_tmap(&tmAt);
      prefetch_tmap(&tmMt);
      int s = 0;
      uint32_t ph = 0, armed = 0, last_ph = 0;
      bool ok = true;
      for (int it = 0; it < L && ok; ++it) {
        for (int p = 0; p < nkx + neb * nsp; ++p) {
          if (!(ok = mbar_wait_sleep(smem_u32(&ctl->bempty[s]), ph ^ 1u, &ctl->abort, bud)))
            break;
          const uint32_t st = bring + s * bsb;
          const uint32_t fb = smem_u32(&ctl->bfull[s]);
          mbar_arrive_expect_tx(fb, bsb);
          if (p < nkx) {
            tma_load_2d(st, &tmAt, p * 64, 0, fb);
          } else {
            const int jj = p - nkx, eb = jj / nsp, sp = jj - eb * nsp;
            tma_load_2d(st, &tmMt, eb * 64, sp * a.r, fb);
          }
          armed |= 1u << s;
          last_ph = (last_ph & ~(1u << s)) | (ph << s);
          if (++s == nb) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        give_up(ctl, a.err);
        for (int k = 0; k < nb; ++k)
          if ((armed >> k) & 1u) drain_wait(smem_u32(&ctl->bfull[k]), (last_ph >> k) & 1u, kDrainNs);
      }
    }
  } else if (warp == 2) {
    // ------------------------- distance-product issuer and codebook producer
    // Lane 0 serves the two warp sets' step streams, each with its own two
    // codebook stages (set j: stages 2j, 2j + 1, alternating between its
    // steps), so neither set waits for the other's books.  Per set: load the
    // next book once its stage is released, and issue the next 128-code chunk
    // of the distance product once the step's operand is written, its book
    // has landed and the chunk's TMEM slot has been read.  Non-blocking
    // probes, a short sleep when nothing can move.
    if constexpr (vq) if (lane == 0) {
      prefetch_tmap(&tmC);
      prefetch_tmap(&tmH);
      constexpr int kStepsC = GD / 16;
      constexpr int kRowB = 2 * GD;
      const int nch = a.K / kChunk;
      const uint32_t total = static_cast<uint32_t>(L * a.R * NGW);   // steps per set
      const uint32_t idd = idesc_bf16(kTile, kChunk);
      const uint32_t cbytes = static_cast<uint32_t>(a.K * a.gd) * 2u;   // codes; the norm rows follow
      const uint32_t hbytes = static_cast<uint32_t>(a.K) * 32u;
      const uint64_t od = narrow_desc<32>(ones);
      uint32_t lb[2] = {0u, 0u};           // books loaded
      int lb_rho[2] = {0, 0}, lb_gi[2] = {0, 0};
      uint32_t x[2] = {0u, 0u};            // chunks issued
      uint32_t st[2] = {0u, 0u};           // step of chunk x
      int ch[2] = {0, 0};                  // chunk of x within its step
      bool got_op[2] = {false, false}, got_cb[2] = {false, false};
      bool issued = false, ok = true;
      uint64_t last = global_ns();
      uint32_t idle = 0;
      while (ok && (st[0] < total || st[1] < total)) {
        bool moved = false;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          // next book of set j
          if (lb[j] < total) {
            const int s = 2 * j + static_cast<int>(lb[j] & 1u);
            if (mbar_test(smem_u32(&ctl->cempty[s]), ((lb[j] >> 1) & 1u) ^ 1u)) {
              const uint32_t fb = smem_u32(&ctl->cfull[s]);
              mbar_arrive_expect_tx(fb, cbytes + hbytes);
              const int row0 = (lb_rho[j] * a.G + 2 * lb_gi[j] + j) * a.K;
              tma_load_2d(cring + s * cbsb, &tmC, 0, row0, fb);
              tma_load_2d(cring + s * cbsb + cbytes, &tmH, 0, row0, fb);
              ++lb[j];
              if (++lb_gi[j] == NGW) {
                lb_gi[j] = 0;
                if (++lb_rho[j] == a.R) lb_rho[j] = 0;
              }
              moved = true;
            }
          }
          // next chunk of set j
          if (st[j] < total) {
            const uint32_t oslot = st[j] & 1u;
            const int s = 2 * j + static_cast<int>(st[j] & 1u);
            if (!got_op[j])
              got_op[j] = mbar_test(smem_u32(&ctl->opready[2 * j + oslot]), (st[j] >> 1) & 1u);
            if (!got_cb[j]) got_cb[j] = mbar_test(smem_u32(&ctl->cfull[s]), (st[j] >> 1) & 1u);
            const uint32_t ds = static_cast<uint32_t>(j);   // one chunk slot per set
            if (got_op[j] && got_cb[j] &&
                mbar_test(smem_u32(&ctl->dempty[ds]), (x[j] & 1u) ^ 1u)) {
              tc_fence_after();
              const uint32_t at = tbase + kColOp + (2u * j + oslot) * 32u;
              const uint32_t dt = tbase + kColDist + ds * kChunk;
              const uint32_t sb = cring + static_cast<uint32_t>(s) * cbsb;
              const uint64_t bd = narrow_desc<(GD == 32 ? 64 : 32)>(
                  sb + static_cast<uint32_t>(ch[j] * kChunk * kRowB));
              const uint64_t hd = narrow_desc<32>(sb + cbytes + static_cast<uint32_t>(ch[j] * kChunk * 32));
              // t = ||c||^2 / 2 (ones x norm rows) - u_hi.c - u_lo.c
              mma_bf16(dt, od, hd, idd, 0u);
#pragma unroll
              for (int k = 0; k < 2 * kStepsC; ++k)
                mma_bf16_ta(dt, at + 8 * k, bd + 2 * (k % kStepsC), idd, 1u);
              mma_commit(smem_u32(&ctl->dfull[ds]));
              issued = true;
              moved = true;
              ++x[j];
              if (++ch[j] == nch) {
                ch[j] = 0;
                ++st[j];
                got_op[j] = got_cb[j] = false;
              }
            }
          }
        }
        if (moved) {
          idle = 0;
          continue;
        }
        __nanosleep(100);
        if ((++idle & 63u) == 0u) {
          const uint64_t now = global_ns();
          if (idle == 64u) last = now;
          if (ctl->abort || now - last > bud) ok = false;
        }
      }
      if (!ok) give_up(ctl, a.err);
      // every product issued has completed before TMEM can be freed, and no
      // book load is still landing
      if (issued) {
        mma_commit(smem_u32(&ctl->vqdone));
        drain_wait(smem_u32(&ctl->vqdone), 0u, ok ? bud : kDrainNs);
      }
      if (!ok) {
        for (int j = 0; j < 2; ++j)
          for (uint32_t b = lb[j] > 2u ? lb[j] - 2u : 0u; b < lb[j]; ++b)
            drain_wait(smem_u32(&ctl->cfull[2 * j + static_cast<int>(b & 1u)]), (b >> 1) & 1u,
                       kDrainNs);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------- projection MMA issuer
    // Lane 0 issues the projection of every tile into the Z accumulator:
    // per 64-column block one X stage (or the gathered anchor rows, held for
    // all -M^T splits of the block) against one B stage.  The VQ distance
    // products are issued by warp 2.
    if (lane == 0) {
      const uint32_t idz = idesc_bf16(kTile, a.r);
      const uint64_t xd0 = sw128_desc(xring);
      const uint64_t bd0 = sw128_desc(bring);
      const int pj_items = nkx + neb * nsp;
      int xs = 0, bs = 0;
      uint32_t xph = 0, bph = 0;
      bool ok = true, issued = false;
      for (int it = 0; it < L && ok; ++it) {
        const int zb = nz == 2 ? (it & 1) : 0;
        const uint32_t zuse = static_cast<uint32_t>(nz == 2 ? (it >> 1) : it);
        if (!(ok = mbar_wait_sleep(smem_u32(&ctl->zempty[zb]), (zuse & 1u) ^ 1u, &ctl->abort,
                                   bud)))
          break;
        tc_fence_after();
        const uint32_t dz = tbase + zb * a.r;
        int sp = 0;
        for (int p = 0; p < pj_items; ++p) {
          if (!(ok = mbar_wait_sleep(smem_u32(&ctl->xfull[xs]), xph, &ctl->abort, bud))) break;
          if (!(ok = mbar_wait_sleep(smem_u32(&ctl->bfull[bs]), bph, &ctl->abort, bud))) break;
          tc_fence_after();
          const uint64_t ad = xd0 + ((static_cast<uint32_t>(xs) * kXBytes) >> 4);
          const uint64_t bd = bd0 + ((static_cast<uint32_t>(bs) * bsb) >> 4);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(dz, ad + 2 * k, bd + 2 * k, idz, (p | k) != 0 ? 1u : 0u);
          issued = true;
          mma_commit(smem_u32(&ctl->bempty[bs]));
          if (++bs == nb) {
            bs = 0;
            bph ^= 1u;
          }
          // an anchor block's rows serve all its -M splits
          bool release_x = true;
          if (p >= nkx) {
            release_x = ++sp == nsp;
            if (release_x) sp = 0;
          }
          if (release_x) {
            mma_commit(smem_u32(&ctl->xempty[xs]));
            if (++xs == nx) {
              xs = 0;
              xph ^= 1u;
            }
          }
        }
        if (ok) mma_commit(smem_u32(&ctl->zfull[zb]));
      }
      if (!ok) give_up(ctl, a.err);
      // every product issued has completed before TMEM can be freed
      if (issued) {
        mma_commit(smem_u32(&ctl->mmadone));
        drain_wait(smem_u32(&ctl->mmadone), 0u, ok ? bud : kDrainNs);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3, j = (warp - kEpiWarp0) >> 2;
    if constexpr (vq) {
      epilogue_vq<GD, NGW>(a, ctl, rg, tbase, base + cring_off, cbsb, q, j, lane);
    } else {
      const uint32_t lanebase = static_cast<uint32_t>(q * 32) << 16;
      const int half = a.r / 2;
      for (int it = 0; it < L; ++it) {
        const int zb = it & 1;
        const uint32_t zuse = static_cast<uint32_t>(it >> 1);
        if (!warp_wait(smem_u32(&ctl->zfull[zb]), zuse & 1u, ctl, bud)) {
          give_up(ctl, a.err);
          break;
        }
        tc_fence_after();
        const int row = q * 32 + lane;
        const int n = rg.t0(it) + row;
        const bool store = row < rg.cnt(it);
        bool bad = false;
        if (store && a.anchor) {
          const int t = a.tids[n];
          bad = t < 0 || t >= a.V;
          if (bad && j == 0) atomicOr(a.err, kErrBadToken);
        }
        const uint32_t tz = tbase + lanebase + zb * a.r;
        for (int c0 = j * half; c0 < (j + 1) * half; c0 += 32) {
          float v[32];
          tmem_ld32(tz + c0, v);
          tmem_wait_ld();
          if (!store) continue;
          if (bad) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
          }
          if (a.mode == kModeZ32) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) +
                                                    static_cast<size_t>(n) * a.r + c0);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) +
                                                  static_cast<size_t>(n) * a.r + c0);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]),
                                  pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                  pack_bf16x2(v[8 * i + 4], v[8 * i + 5]),
                                  pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->zempty[zb]));
      }
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

template <int GD, int NGW>
cudaError_t launch_one(const CUtensorMap& tmX, const CUtensorMap& tmAt, const CUtensorMap& tmMt,
                       const CUtensorMap& tmC, const CUtensorMap& tmH, const CUtensorMap& tmE,
                       const CompressArgs& a, uint32_t smem, int grid, cudaStream_t s) {
  const cudaError_t e = set_smem(k_compress_pipe<GD, NGW>, smem);
  if (e != cudaSuccess) return e;
  return launch_chained(k_compress_pipe<GD, NGW>, dim3(grid), dim3(kThreads), smem, s, tmX, tmAt,
                        tmMt, tmC, tmH, tmE, a);
}

}  // namespace

uint32_t compress_pipe_ctl_bytes() { return static_cast<uint32_t>(sizeof(Ctl)); }
uint32_t compress_pipe_ones_bytes() { return kOnesBytes; }

bool compress_pipe_supported(int r, bool vq, int gd, int G, int K) {
  if (!vq) return r % 64 == 0 && r <= 256;
  if (r != 64 && r != 128) return false;
  if (K % kChunk != 0) return false;
  if (gd != 16 && gd != 32) return false;
  const int ngw = G / 2;
  return G % 2 == 0 && (ngw == 1 || ngw == 2 || ngw == 4) && ngw * gd * 2 == r;
}

cudaError_t launch_compress_pipe(const CUtensorMap& tmX, const CUtensorMap& tmAt,
                                 const CUtensorMap& tmMt, const CUtensorMap& tmC,
                                 const CUtensorMap& tmH, const CUtensorMap& tmE,
                                 const CompressArgs& a, uint32_t smem_bytes, int grid,
                                 cudaStream_t s) {
  if (a.mode != kModeVQ)
    return launch_one<0, 1>(tmX, tmAt, tmMt, tmC, tmH, tmE, a, smem_bytes, grid, s);
  const int ngw = a.G / 2;
  if (a.gd == 32 && ngw == 2)
    return launch_one<32, 2>(tmX, tmAt, tmMt, tmC, tmH, tmE, a, smem_bytes, grid, s);
  if (a.gd == 16 && ngw == 4)
    return launch_one<16, 4>(tmX, tmAt, tmMt, tmC, tmH, tmE, a, smem_bytes, grid, s);
  if (a.gd == 32 && ngw == 1)
    return launch_one<32, 1>(tmX, tmAt, tmMt, tmC, tmH, tmE, a, smem_bytes, grid, s);
  if (a.gd == 16 && ngw == 2)
    return launch_one<16, 2>(tmX, tmAt, tmMt, tmC, tmH, tmE, a, smem_bytes, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace mapl
