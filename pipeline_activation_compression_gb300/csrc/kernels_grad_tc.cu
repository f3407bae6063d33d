// kernels_grad_tc.cu -- Euclidean gradient of the projector A on the tensor
// cores (backward pass of the codec, MAPL §3.2; the gradient that §3.3's SPEL
// step consumes).
//
// With X_res = X - anchor, Z the payload and gZ = dL/dX_hat A:
//     dA = X_res^T gZ + dL/dX_hat^T Z                                (d x r)
// factored anchor (E[tids] P):  dA = X^T gZ + gXh^T Z - P^T (E[tids]^T gZ)
// first-boundary anchor:        dA = X^T gZ + gXh^T Z - E_emb[tids]^T gZ
//
// The tensor cores compute the transpose, dA^T = gZ^T X + Z^T gXh (M = r,
// N = a slab of W = 256 columns of d): every product contracts over the
// tokens, the row index of the row-major inputs, so both operands are
// MN-major (128-byte swizzle: 64 elements of M or N per 128-byte row, one
// row per token, 8-token groups 1 KB apart, consecutive 64-element atoms one
// TMA box apart), and N = 256 keeps the tensor pipe busy through the
// per-block commit that a 128-wide N leaves exposed.
//
// k_grad: one cooperative launch, one CTA per SM, in three phases.
//  1. Tiles.  CTA (tile, split) accumulates the partial of its column tile
//     over its token split in TMEM: X tiles (W columns of d: gZ^T X + Z^T
//     gXh) and E tiles (W columns of the anchor table, gathered by token id:
//     gZ^T E[tids]; columns of r for the factored anchor when r > 128,
//     columns of d for the embedding anchor).  When r <= 128 the factored
//     anchor's product gZ^T E[tids] (r x r) is folded into the X tiles: each
//     takes every nX-th token block of its split into a second accumulator.
//     The drain stores each partial in dA's own layout (column c of the
//     tile, TMEM lane a: element [c][a]), so a warp's stores are coalesced.
//  2. After a grid barrier, T = E[tids]^T gZ is summed from its partials.
//  3. After a second barrier, dA = sum of the X partials minus the anchor
//     term (the E partials, or P^T T).
// Every sum runs in a fixed order, so the result does not depend on timing.
//
// Phase 1 streams one stage per 32-token block: [B1 | B2 | A1 | A2] =
// [X or gathered E slab | gXh slab | gZ | Z], each slab one 3-D TMA box
// (64 elements x 32 tokens x its 64-element atoms) so that a block costs
// four TMA instructions.  The folded anchor's rows go through a two-stage
// ring of their own, gathered by a warp of their own so that the producer's
// stream of boxes never waits for a token id.  Warp 0: TMA producer; warp 1:
// TMEM and the MMA issuer; warps 2..5: drain; warp 6: the folded rows.  Waits are bounded; a
// CTA that gives up sets the error word, still joins both grid barriers
// (whose own waits are bounded too) and unwinds.
#include "mapl_internal.h"
#include "ptx.cuh"

namespace mapl {

namespace {

constexpr int kGThreads = 256;
constexpr int kNF = 4;   // stages of the folded-gather ring
constexpr int kBatch = 20;   // loads in flight per thread in the reductions
constexpr uint32_t kFullMask = 0xffffffffu;

struct GCtl {
  uint64_t full[kGradMaxStages], empty[kGradMaxStages];
  uint64_t fullF[kNF], emptyF[kNF];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
};

// Shared-memory descriptor of an MN-major operand in the 128-byte swizzled
// layout TMA writes for a box of {64 elements, rows}: `atom` bytes between
// consecutive 64-element atoms of M or N, 1 KB between 8-row groups of K.
__device__ __forceinline__ uint64_t mn_desc(uint32_t addr, uint32_t atom) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((atom >> 4) & 0x3FFFu) << 16;   // leading: next MN atom
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                // stride: next 8 K rows
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;                        // swizzle 128 B
  return d;
}

// kind::f16 instruction descriptor, bf16 A and B both MN-major, fp32 D.
__host__ __device__ constexpr uint32_t idesc_mn_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void g_give_up(GCtl* c, int* err) {
  c->abort = 1;
  atomicOr(err, kErrTimeout);
}

__device__ __forceinline__ void g_drain(uint32_t bar, uint32_t parity, uint64_t budget) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > budget) return;
}

// A producer's ring position and the record of what it may still have in
// flight when it gives up.
struct Ring {
  int s = 0;
  uint32_t ph = 0, armed = 0, last_ph = 0;
  __device__ void advance(int n) {
    armed |= 1u << s;
    last_ph = (last_ph & ~(1u << s)) | (ph << s);
    if (++s == n) {
      s = 0;
      ph ^= 1u;
    }
  }
  __device__ void drain(uint64_t* full, int n) const {
    for (int k = 0; k < n; ++k)
      if ((armed >> k) & 1u) g_drain(smem_u32(&full[k]), (last_ph >> k) & 1u, 10000000ull);
  }
};

// Grid-wide barrier over a counter zeroed before the launch: barrier k of
// the launch completes when the counter reaches k * gridDim.x (the launch is
// cooperative, so every CTA is resident).  The wait is bounded; a CTA that
// gives up sets the error word and goes on.
__device__ void grid_barrier(unsigned int* bar, unsigned int k, int* err, uint64_t budget) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
    const unsigned int target = k * gridDim.x;
    const uint64_t t0 = global_ns();
    while (true) {
      unsigned int v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar) : "memory");
      if (v >= target) break;
      if (global_ns() - t0 > budget) {
        atomicOr(err, kErrTimeout);
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
  }
  __syncthreads();
}

__device__ __forceinline__ void add4(float4& s, const float4& v) {
  s.x += v.x;
  s.y += v.y;
  s.z += v.z;
  s.w += v.w;
}

__global__ void __launch_bounds__(kGThreads, 1)
    k_grad(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmGX,
           const __grid_constant__ CUtensorMap tmGZ, const __grid_constant__ CUtensorMap tmZ,
           const __grid_constant__ CUtensorMap tmE, const GradArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x / a.S, split = blockIdx.x - tile * a.S;
  const bool xtile = tile < a.nX;
  const bool fold = a.fold && xtile;
  const int W = a.W;
  const int col0 = (xtile ? tile : tile - a.nX) * W;      // first column of this tile
  const int kb = a.kb;                                    // tokens per block
  const uint32_t atom = static_cast<uint32_t>(kb) * 128u; // one box: 64 elements x kb rows
  const int nB = W / 64;                                  // B atoms per operand
  const int nA = a.nM * 2;                                // A atoms per operand (2 per M block)
  const int nFa = a.r <= 64 ? 1 : 2;                      // atoms of a folded gather (N = r)
  // stage: [B1 (nB) | B2 (nB) | A1 (nA) | A2 (nA)]
  const uint32_t offB2 = nB * atom, offA1 = 2 * nB * atom, offA2 = (2 * nB + nA) * atom;
  const uint32_t sbytes = (2 * nB + 2 * nA) * atom, fbytes = 2 * atom;
  const uint32_t ring = smem_u32(base), ringF = ring + a.nstage * sbytes;
  GCtl* ctl = reinterpret_cast<GCtl*>(base + a.nstage * sbytes + kNF * fbytes);
  const int nkb_all = (a.N + kb - 1) / kb;
  const int kb0 = static_cast<int>(static_cast<long long>(nkb_all) * split / a.S);
  const int kb1 = static_cast<int>(static_cast<long long>(nkb_all) * (split + 1) / a.S);
  const int nblk = kb1 - kb0;
  auto has_e = [&](int q) { return fold && q % a.nX == tile; };
  const uint64_t bud = a.timeout_ns;
  const int ncols = a.nM * W + (fold ? a.r : 0);
  uint32_t tcols = 32;   // a power of two >= ncols
  while (tcols < static_cast<uint32_t>(ncols)) tcols <<= 1;

  if (threadIdx.x == 0) {
    for (int k = 0; k < a.nstage; ++k) {
      mbar_init(smem_u32(&ctl->full[k]), 1);
      mbar_init(smem_u32(&ctl->empty[k]), 1);
    }
    for (int k = 0; k < kNF; ++k) {
      mbar_init(smem_u32(&ctl->fullF[k]), 1);
      mbar_init(smem_u32(&ctl->emptyF[k]), 1);
    }
    mbar_init(smem_u32(&ctl->done), 1);
    ctl->abort = 0;
    fence_mbar_init();
    fence_async_shared();
  }
  if (warp == 1) tmem_alloc(smem_u32(&ctl->tmem_base), tcols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ctl->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    // An E tile's rows: lane L issues four-row gather L of a block (atom
    // L / (kb / 4), rows 4 (L % (kb / 4)) ..).  A block's ids are loaded when
    // the previous block's gathers are issued and checked only when their
    // own are, so the load's latency overlaps a block.  Ids outside [0, V)
    // and tokens past N read row V, outside the table, which TMA fills with
    // zeros.
    const int rr = (lane % (kb / 4)) * 4;
    const int gat = nB * (kb / 4);   // lanes that gather
    int ids[4] = {0, 0, 0, 0};
    auto load_ids = [&](int q) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int n = (kb0 + q) * kb + rr + k;
        ids[k] = n < a.N ? __ldg(a.tids + n) : a.V;
      }
    };
    if (!xtile && nblk > 0 && lane < gat) load_ids(0);
    Ring rg;
    bool ok = true;
    for (int q = 0; q < nblk; ++q) {
      const int t0 = (kb0 + q) * kb;
      if (!(ok = __all_sync(kFullMask, mbar_wait_sleep(smem_u32(&ctl->empty[rg.s]), rg.ph ^ 1u,
                                                       &ctl->abort, bud))))
        break;
      const uint32_t st = ring + rg.s * sbytes;
      const uint32_t fb = smem_u32(&ctl->full[rg.s]);
      if (lane == 0) {
        mbar_arrive_expect_tx(fb, (xtile ? 2 * nB + 2 * nA : nB + nA) * atom);
        if (xtile) {
          tma_load_3d(st, &tmX, 0, t0, col0 / 64, fb);
          tma_load_3d(st + offB2, &tmGX, 0, t0, col0 / 64, fb);
        }
        // A atoms past r (r = 64: the second) lie outside the tensor: zeros
        tma_load_3d(st + offA1, &tmGZ, 0, t0, 0, fb);
        if (xtile) tma_load_3d(st + offA2, &tmZ, 0, t0, 0, fb);
      }
      __syncwarp();
      if (!xtile && lane < gat) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (ids[k] < 0 || ids[k] >= a.V) {
            if (t0 + rr + k < a.N && lane < kb / 4) atomicOr(a.err, kErrBadToken);
            ids[k] = a.V;
          }
        const int h = lane / (kb / 4);
        tma_gather4(st + h * atom + rr * 128, &tmE, col0 + 64 * h, ids[0], ids[1], ids[2], ids[3],
                    fb);
        if (q + 1 < nblk) load_ids(q + 1);
      }
      rg.advance(a.nstage);
    }
    if (!ok) {
      if (lane == 0) g_give_up(ctl, a.err);
      rg.drain(ctl->full, a.nstage);
    }
  } else if (warp == 6) {
    // -------------------------------------------------- folded anchor's rows
    // Four-row TMA gathers into the F ring: lane L < 2 kb / 4 issues gather
    // L of a block (atom L / (kb / 4), rows 4 (L % (kb / 4)) ..).  Ids are
    // loaded two folded blocks ahead and checked when their gathers are
    // issued; ids outside [0, V) and tokens past N read row V, outside the
    // table, which TMA fills with zeros.
    if (fold) {
      const int rr = (lane % (kb / 4)) * 4;
      const int gat = nFa * (kb / 4);
      auto next_e = [&](int q) {
        while (q < nblk && !has_e(q)) ++q;
        return q;
      };
      auto load_ids = [&](int q, int (&ids)[4]) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int n = (kb0 + q) * kb + rr + k;
          ids[k] = (q < nblk && n < a.N && lane < gat) ? __ldg(a.tids + n) : a.V;
        }
      };
      int q0 = next_e(0), q1 = next_e(q0 + 1);
      int ids0[4], ids1[4];
      load_ids(q0, ids0);
      load_ids(q1, ids1);
      Ring rf;
      bool ok = true;
      while (q0 < nblk) {
        if (!(ok = __all_sync(kFullMask, mbar_wait_sleep(smem_u32(&ctl->emptyF[rf.s]), rf.ph ^ 1u,
                                                         &ctl->abort, bud))))
          break;
        const uint32_t ff = smem_u32(&ctl->fullF[rf.s]);
        if (lane == 0) mbar_arrive_expect_tx(ff, nFa * atom);
        __syncwarp();
        if (lane < gat) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (ids0[k] < 0 || ids0[k] >= a.V) {
              if ((kb0 + q0) * kb + rr + k < a.N && lane < kb / 4) atomicOr(a.err, kErrBadToken);
              ids0[k] = a.V;
            }
          const int h = lane / (kb / 4);
          tma_gather4(ringF + rf.s * fbytes + h * atom + rr * 128, &tmE, 64 * h, ids0[0], ids0[1],
                      ids0[2], ids0[3], ff);
        }
        rf.advance(kNF);
        q0 = q1;
#pragma unroll
        for (int k = 0; k < 4; ++k) ids0[k] = ids1[k];
        q1 = next_e(q1 + 1);
        load_ids(q1, ids1);
      }
      if (!ok) {
        if (lane == 0) g_give_up(ctl, a.err);
        rf.drain(ctl->fullF, kNF);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idW = idesc_mn_bf16(128, W), idF = idesc_mn_bf16(128, a.r);
      int s = 0, sf = 0;
      uint32_t ph = 0, phf = 0;
      bool ok = true, issued = false, first_e = true;
      for (int q = 0; ok && q < nblk; ++q) {
        const bool e = has_e(q);
        if (!(ok = mbar_wait_sleep(smem_u32(&ctl->full[s]), ph, &ctl->abort, bud))) break;
        if (e && !(ok = mbar_wait_sleep(smem_u32(&ctl->fullF[sf]), phf, &ctl->abort, bud))) break;
        tc_fence_after();
        const uint32_t st = ring + s * sbytes, fs = ringF + sf * fbytes;
        for (int kk = 0; kk < kb / 16; ++kk) {
          const uint32_t ko = static_cast<uint32_t>(kk) * 2048u;
          const uint32_t acc = (q == 0 && kk == 0) ? 0u : 1u;
          for (int mb = 0; mb < a.nM; ++mb) {
            const uint32_t d0 = tbase + static_cast<uint32_t>(mb * W);
            const uint32_t am = static_cast<uint32_t>(2 * mb) * atom + ko;
            mma_bf16(d0, mn_desc(st + offA1 + am, atom), mn_desc(st + ko, atom), idW, acc);
            if (xtile)
              mma_bf16(d0, mn_desc(st + offA2 + am, atom), mn_desc(st + offB2 + ko, atom), idW, 1u);
          }
          if (e)   // folded anchor (r <= 128): gZ^T E[tids], N = r
            mma_bf16(tbase + static_cast<uint32_t>(W), mn_desc(st + offA1 + ko, atom),
                     mn_desc(fs + ko, atom), idF, (first_e && kk == 0) ? 0u : 1u);
        }
        issued = true;
        mma_commit(smem_u32(&ctl->empty[s]));
        if (++s == a.nstage) {
          s = 0;
          ph ^= 1u;
        }
        if (e) {
          first_e = false;
          mma_commit(smem_u32(&ctl->emptyF[sf]));
          if (++sf == kNF) {
            sf = 0;
            phf ^= 1u;
          }
        }
      }
      if (!ok) g_give_up(ctl, a.err);
      // the accumulators are complete (or, on give-up, every product finished)
      if (issued) mma_commit(smem_u32(&ctl->done));
      else mbar_arrive(smem_u32(&ctl->done));
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------------- drain
    const int qd = warp & 3;
    const bool ok = __all_sync(kFullMask, mbar_wait_sleep(smem_u32(&ctl->done), 0u, &ctl->abort,
                                                          bud + 100000000ull));
    if (ok) {
      tc_fence_after();
      const uint32_t taddr = tbase + (static_cast<uint32_t>(qd * 32) << 16);
      // this tile's partial, element [c][a] = TMEM lane a, column mb W + c
      float* dst = a.ws + static_cast<size_t>(tile * a.S + split) * W * a.r;
      const bool none = nblk == 0;
      for (int mb = 0; mb < a.nM; ++mb) {
        const int ar = mb * 128 + qd * 32 + lane;   // row of r
        for (int c = 0; c < W; c += 32) {
          float v[32];
          tmem_ld32(taddr + static_cast<uint32_t>(mb * W + c), v);
          tmem_wait_ld();
          if (ar < a.r) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              dst[static_cast<size_t>(c + i) * a.r + ar] = none ? 0.f : v[i];
          }
        }
      }
      if (fold) {
        // folded anchor partial: lane j, column a -> T partial [a][j]
        float* dT = a.wsT + static_cast<size_t>(tile * a.S + split) * a.r * a.r;
        const int j = qd * 32 + lane;
        const bool nonet = tile >= nblk;   // no block of this split fell to this tile
        for (int c = 0; c < a.r; c += 32) {
          float v[32];
          tmem_ld32(taddr + static_cast<uint32_t>(W + c), v);
          tmem_wait_ld();
          if (j < a.r) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              dT[static_cast<size_t>(c + i) * a.r + j] = nonet ? 0.f : v[i];
          }
        }
      }
    } else if (lane == 0) {
      g_give_up(ctl, a.err);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tbase, tcols);
  }

  // ------------------------------------------------- phase 2: T from partials
  grid_barrier(a.bar, 1u, a.err, bud + 100000000ull);
  const int w8 = warp;                              // 8 warps
  float4* red = reinterpret_cast<float4*>(base);    // [8][32]: the ring is free now
  if (!a.emb) {
    // a unit is 128 consecutive values of T (one float4 per lane); partial p
    // of the unit starts at src + p * pstride + ub
    const int nunits = a.r * a.r / 128;
    const float* src;
    size_t pstride;
    int np;
    if (a.fold) {
      src = a.wsT;
      pstride = static_cast<size_t>(a.r) * a.r;
      np = a.nX * a.S;
    } else {
      src = a.ws + static_cast<size_t>(a.nX) * a.S * W * a.r;
      pstride = static_cast<size_t>(W) * a.r;
      np = a.S;
    }
    const size_t ps4 = pstride / 4;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
      const int e0 = u * 128;   // first element of T in this unit
      size_t ub;
      if (a.fold) {
        ub = static_cast<size_t>(e0) + lane * 4;
      } else {   // row ta of T: row ta % W of E tile ta / W (one unit lies in one row)
        const int ta = e0 / a.r, tj = e0 % a.r + lane * 4;
        ub = static_cast<size_t>(ta / W) * a.S * W * a.r + static_cast<size_t>(ta % W) * a.r + tj;
      }
      const float4* b4 = reinterpret_cast<const float4*>(src + ub);
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int p0 = w8; p0 < np; p0 += 8 * kBatch) {
        float4 v[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
          v[k] = p0 + 8 * k < np ? __ldcg(b4 + (p0 + 8 * k) * ps4) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < kBatch; ++k) add4(s, v[k]);
      }
      red[w8 * 32 + lane] = s;
      __syncthreads();
      if (w8 == 0) {
        float4 t = red[lane];
#pragma unroll
        for (int k = 1; k < 8; ++k) add4(t, red[k * 32 + lane]);
        __stcg(reinterpret_cast<float4*>(a.T + e0) + lane, t);
      }
      __syncthreads();
    }
  }

  // --------------------------------------- phase 3: dA = sum - anchor term
  grid_barrier(a.bar, 2u, a.err, bud + 100000000ull);
  {
    // a unit is 8 rows of dA (warp w: row i0 + w) by 128 columns (a float4
    // per lane).  For the factored anchor, T's rows a0..a0+127 (the unit's
    // 128 columns) and P's rows a0..a0+127 (the unit's 8 columns) are copied
    // to shared memory by cp.async, the first slice before the split sums
    // so that both are in flight together.
    const uint32_t sT = smem_u32(base);                 // [128][32] float4
    const uint32_t sPb = sT + 128 * 32 * 16;            // [128][8] bf16
    const float4* sT4 = reinterpret_cast<const float4*>(base);
    const __nv_bfloat16* sP = reinterpret_cast<const __nv_bfloat16*>(base + 128 * 32 * 16);
    const int njb = (a.r + 127) / 128;
    const int nunits = (a.d + 7) / 8 * njb;
    const size_t pst4 = static_cast<size_t>(W) * a.r / 4;          // one split's partial
    const size_t eoff4 = static_cast<size_t>(a.nX) * a.S * pst4;   // the E tiles' partials
    for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
      const int i0 = (u / njb) * 8, jb = u % njb;
      const int i = i0 + w8, j = jb * 128 + lane * 4;
      const bool live = i < a.d && j < a.r;
      const int nc4 = (a.r - jb * 128) / 4 < 32 ? (a.r - jb * 128) / 4 : 32;   // float4 columns
      auto stage = [&](int a0) {
        const int na = a.r - a0 < 128 ? a.r - a0 : 128;
        for (int x = threadIdx.x; x < na * 32; x += kGThreads) {
          const int row = x >> 5, c = x & 31;
          if (c < nc4)
            cp_async16(sT + static_cast<uint32_t>(row * 512 + c * 16),
                       a.T + static_cast<size_t>(a0 + row) * a.r + jb * 128 + c * 4);
        }
        for (int x = threadIdx.x; x < na; x += kGThreads)
          cp_async16(sPb + static_cast<uint32_t>(x * 16), a.P + static_cast<size_t>(a0 + x) * a.d + i0);
      };
      if (!a.emb) stage(0);
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      if (live) {
        const float4* b4 = reinterpret_cast<const float4*>(
            a.ws + (static_cast<size_t>(i / W) * a.S * W + i % W) * a.r + j);
        for (int sp0 = 0; sp0 < a.S; sp0 += kBatch) {
          float4 v[kBatch];
#pragma unroll
          for (int k = 0; k < kBatch; ++k)
            v[k] = sp0 + k < a.S ? __ldcg(b4 + (sp0 + k) * pst4) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int k = 0; k < kBatch; ++k) add4(s, v[k]);
          if (a.emb) {
#pragma unroll
            for (int k = 0; k < kBatch; ++k)
              v[k] = sp0 + k < a.S ? __ldcg(b4 + eoff4 + (sp0 + k) * pst4)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
              s.x -= v[k].x;
              s.y -= v[k].y;
              s.z -= v[k].z;
              s.w -= v[k].w;
            }
          }
        }
      }
      if (!a.emb) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int a0 = 0; a0 < a.r; a0 += 128) {
          cp_async_wait_all();
          __syncthreads();
          const int na = a.r - a0 < 128 ? a.r - a0 : 128;
#pragma unroll 8
          for (int aa = 0; aa < na; ++aa) {
            const float p = __bfloat162float(sP[aa * 8 + w8]);
            const float4 t = sT4[aa * 32 + lane];
            acc.x = fmaf(p, t.x, acc.x);
            acc.y = fmaf(p, t.y, acc.y);
            acc.z = fmaf(p, t.z, acc.z);
            acc.w = fmaf(p, t.w, acc.w);
          }
          __syncthreads();   // the slice is no longer read
          if (a0 + 128 < a.r) stage(a0 + 128);
        }
        s.x -= acc.x;
        s.y -= acc.y;
        s.z -= acc.z;
        s.w -= acc.w;
      }
      if (live) *reinterpret_cast<float4*>(a.dA + static_cast<size_t>(i) * a.r + j) = s;
    }
  }
}

}  // namespace

uint32_t grad_stage_bytes(int r, int W, int kb) {
  const int nA = 2 * ((r + 127) / 128);
  return static_cast<uint32_t>(2 * (W / 64) + 2 * nA) * static_cast<uint32_t>(kb) * 128u;
}

uint32_t grad_fring_bytes(int kb) { return kNF * 2u * static_cast<uint32_t>(kb) * 128u; }

uint32_t grad_ctl_bytes() { return static_cast<uint32_t>(sizeof(GCtl)); }

cudaError_t launch_grad_A(const CUtensorMap& tmX, const CUtensorMap& tmGX, const CUtensorMap& tmGZ,
                          const CUtensorMap& tmZ, const CUtensorMap& tmE, const GradArgs& a,
                          int grid, uint32_t smem, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(k_grad, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(a.bar, 0, sizeof(unsigned int), s)) != cudaSuccess) return e;
  void* args[] = {const_cast<CUtensorMap*>(&tmX), const_cast<CUtensorMap*>(&tmGX),
                  const_cast<CUtensorMap*>(&tmGZ), const_cast<CUtensorMap*>(&tmZ),
                  const_cast<CUtensorMap*>(&tmE), const_cast<GradArgs*>(&a)};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k_grad), dim3(grid),
                                     dim3(kGThreads), args, smem, s);
}

}  // namespace mapl
