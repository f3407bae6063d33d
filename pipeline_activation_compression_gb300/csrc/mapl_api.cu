// mapl_api.cu -- host side of the C ABI declared in include/mapl.h: argument
// validation, plan memory and operand layouts, TMA descriptors, launches.
#include <cublas_v2.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>
#include <algorithm>

#include "mapl_internal.h"

using namespace mapl;

struct mapl_plan_s {
  mapl_config cfg{};
  int device = 0;
  int num_sms = 0;
  bool vq = false;
  bool tc = false;        // bf16 tensor-core path
  int gd = 0;
  PlanDevice p;
  CUtensorMap tmAt{}, tmMt{}, tmC{}, tmH{}, tmB{};
  uint64_t timeout_ns = kDefaultTimeoutNs;
  // launch geometry
  int c_nstage = 0;
  uint32_t c_stage = 0, c_smem = 0;
  int d_nstage = 0;
  uint32_t d_stage = 0, d_smem = 0, d_abytes = 0, d_nc = 0;
  bool d_stream = false;
  int d_nab = 0;                      // > 0: persistent kernel with d_nab A buffers
  // pipelined compress kernel (shapes it supports), else the ring kernel above
  bool c_pipe = false;
  int p_nx = 0, p_nb = 0, p_ncb = 0;
  uint32_t p_bstage = 0, p_cstage = 0, p_smem = 0;
  // cuBLAS handle for the plan-time products (M = P_send A and the
  // first-boundary table E_emb A), made on first use
  cublasHandle_t blas = nullptr;
  // sender anchor: E_send[tids] P_send (re = r, three -M terms), or with
  // mapl_plan_set_embedding_anchor the first-boundary E_emb[tids] (re = 3r,
  // one term): table [hi|mid|lo] of E_emb A and -[I; I; I]
  int re = 0, nsplit = kNumSplit;
  const void* E_emb = nullptr;
  void* emb_pool = nullptr;           // [T fp32 V x r | table V x 3r bf16 | M r x 3r bf16]
  float* emb_T = nullptr;
  __nv_bfloat16* emb_tab = nullptr;
  CUtensorMap tmMt_emb{};
  // gradient codebooks (MCVQ of backward gradients): [Cb R x G x K x gd bf16
  // | norm rows R x G x K x 16 bf16 | cnorm | cmax] in one allocation, and
  // their tensor maps
  void* gpool = nullptr;
  __nv_bfloat16* Cb_g = nullptr;
  __nv_bfloat16* Hs_g = nullptr;
  float* cnorm_g = nullptr;
  float* cmax_g = nullptr;
  CUtensorMap tmC_g{}, tmH_g{};
};

namespace {

thread_local std::string g_last_error;

mapl_status fail(mapl_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

mapl_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MAPL_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elt_size(const mapl_config& c) { return c.dtype == MAPL_BF16 ? 2 : 4; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major (outer x inner) matrix, 128-byte
// swizzled boxes of box_outer rows x 64 elements; out-of-range reads are zero.
bool make_tmap(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
               uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D bf16 tensor map viewing a row-major (outer x inner) matrix as
// {64 elements, outer rows, inner / 64 atoms}: one box of {64, box_outer,
// box_atoms} lands in shared memory as box_atoms consecutive 128-byte
// swizzled atoms of box_outer rows (atoms past the matrix read zeros).
bool make_tmap_atoms(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                     uint32_t box_outer, uint32_t box_atoms) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, outer, inner / 64};
  cuuint64_t strides[2] = {inner * 2, 128};
  cuuint32_t box[3] = {64, box_outer, box_atoms};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

constexpr uint32_t kSmemMax = 232448;   // opt-in dynamic shared memory per CTA

mapl_status validate(const mapl_config* c) {
  if (!c) return fail(MAPL_ERR_INVALID_ARG, "config is NULL");
  if (c->dtype != MAPL_F32 && c->dtype != MAPL_BF16)
    return fail(MAPL_ERR_INVALID_ARG, "dtype must be MAPL_F32 or MAPL_BF16");
  if (c->flags != 0) return fail(MAPL_ERR_INVALID_ARG, "flags must be 0");
  if (c->d < 64 || c->d % 64 != 0 || c->d > (1 << 16))
    return fail(MAPL_ERR_INVALID_ARG, "d must be a positive multiple of 64 (<= 65536)");
  if (c->r < 16 || c->r % 16 != 0 || c->r > 512 || c->r > c->d)
    return fail(MAPL_ERR_INVALID_ARG, "r must be a multiple of 16 in [16, min(512, d)]");
  if (c->V < 1 || c->V > 0x7fffffff) return fail(MAPL_ERR_INVALID_ARG, "V must be in [1, 2^31)");
  const bool vq = c->G != 0 || c->R != 0 || c->K != 0;
  if (vq) {
    if (c->G < 1 || c->r % c->G != 0) return fail(MAPL_ERR_INVALID_ARG, "G must divide r");
    if (c->R < 1 || c->R > 8) return fail(MAPL_ERR_INVALID_ARG, "R must be in [1, 8]");
    if (c->K < 1 || c->K > 256) return fail(MAPL_ERR_INVALID_ARG, "K must be in [1, 256]");
  }
  if (c->dtype == MAPL_BF16) {
    if (c->r % 64 != 0)
      return fail(MAPL_ERR_UNSUPPORTED, "bf16 tensor-core path needs r % 64 == 0");
    if (vq) {
      const int64_t gd = c->r / c->G;
      if (gd != 16 && gd != 32)
        return fail(MAPL_ERR_UNSUPPORTED, "bf16 VQ needs group width r/G in {16, 32}");
      if (c->K % 64 != 0)
        return fail(MAPL_ERR_UNSUPPORTED, "bf16 VQ needs K a multiple of 64");
      if (c->r > 256)
        return fail(MAPL_ERR_UNSUPPORTED, "bf16 VQ needs r <= 256");
    }
  }
  return MAPL_OK;
}

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

mapl_status geometry(mapl_plan_s* pl) {
  const mapl_config& c = pl->cfg;
  const uint32_t slack = 1024;
  // compress (persistent): ring of stages + residual operand slots + control
  {
    uint32_t st = 16384u + static_cast<uint32_t>(c.r) * 128u;
    st = (st + 1023u) & ~1023u;
    uint32_t extra = compress_ctl_bytes() + 64 + slack + 2 * 128 * 4;   // + tile ids
    if (pl->vq) {
      extra += 2u * static_cast<uint32_t>(c.K * (c.r / c.G)) * 2u;         // codebook ring
      extra += static_cast<uint32_t>(c.G < 2 ? c.G : 2) * 16384u;         // residual slots
      extra += (static_cast<uint32_t>(c.R * c.G * c.K) * 4u + 15u) & ~15u; // ||c||^2
    }
    int ns = static_cast<int>((kSmemMax - extra) / st);
    if (ns > 8) ns = 8;
    if (ns < 2) return fail(MAPL_ERR_UNSUPPORTED, "compress stages do not fit in shared memory");
    pl->c_nstage = ns;
    pl->c_stage = st;
    pl->c_smem = ns * st + extra;
  }
  // pipelined compress: X ring (HBM), B ring (A^T and -M^T blocks from L2),
  // codebook ring
  pl->c_pipe = compress_pipe_supported(static_cast<int>(c.r), pl->vq, pl->gd, c.G, c.K);
  if (pl->c_pipe) {
    const uint32_t fixed = compress_pipe_ctl_bytes() + 64 + slack +
                           (pl->vq ? compress_pipe_ones_bytes() : 0u);
    const uint32_t bst = static_cast<uint32_t>(c.r) * 128u;
    // a codebook stage: the book's codes, then its K norm rows of 32 bytes
    const uint32_t cst =
        pl->vq ? ((static_cast<uint32_t>(c.K * pl->gd) * 2u + static_cast<uint32_t>(c.K) * 32u +
                   1023u) & ~1023u)
               : 0u;
    const int ncb = pl->vq ? 4 : 0;   // two codebook stages per epilogue warp set
    // without codebooks, half the shared memory goes to the B ring: its
    // blocks are re-read from L2 for every tile, so it needs as many bytes
    // in flight as the X ring
    int nb = bst > 16384u ? 3 : 4;
    if (!pl->vq) {
      nb = static_cast<int>((kSmemMax - fixed) / 2u / bst);
      if (nb > 8) nb = 8;
      if (nb < 3) nb = 3;
    }
    const uint32_t used = fixed + nb * bst + ncb * cst;
    int nx = used < kSmemMax ? static_cast<int>((kSmemMax - used) / 16384u) : 0;
    if (nx > 12) nx = 12;
    if (nx >= 3) {
      pl->p_nx = nx;
      pl->p_nb = nb;
      pl->p_ncb = ncb;
      pl->p_bstage = bst;
      pl->p_cstage = cst;
      pl->p_smem = used + nx * 16384u;
    } else {
      pl->c_pipe = false;
    }
  }
  const uint32_t ctl = decompress_ctl_bytes() + 64;
  // decompress.  r <= 256: persistent kernel, one CTA per SM, the A operand
  // [Z_hat | E'] in TMEM (two buffers when they fit beside the two NC-column
  // accumulators in the 512 columns), shared memory for the [A^T | P'^T]
  // ring, as many stages as fit (at most 12).  Larger r: one CTA per tile,
  // A streamed per stage.
  {
    const uint32_t a_res = static_cast<uint32_t>(2 * c.r / 64) * 16384u;
    pl->d_stream = a_res > 131072u;
    // output columns per accumulator chunk: 128 beside the TMEM-resident A,
    // up to 256 when A is streamed
    const uint32_t NC = pl->d_stream ? ((c.d % 256 == 0) ? 256u : ((c.d % 128 == 0) ? 128u : 64u))
                                     : ((c.d % 128 == 0) ? 128u : 64u);
    pl->d_nc = NC;
    if (!pl->d_stream) {
      const uint32_t acols = static_cast<uint32_t>(c.r);   // K = 2r bf16, two per column
      const int nab = 2 * NC + 2 * acols <= 512u ? 2 : (2 * NC + acols <= 512u ? 1 : 0);
      if (nab == 0) return fail(MAPL_ERR_UNSUPPORTED, "decompress operands do not fit in TMEM");
      const uint32_t extra = decompress_pt_ctl_bytes() + 64 + slack;
      const uint32_t st = 2u * NC * 128u;   // two 64-element K-blocks of NC rows
      int ns = static_cast<int>((kSmemMax - extra) / st);
      if (ns > 12) ns = 12;
      if (ns < 3) return fail(MAPL_ERR_UNSUPPORTED, "decompress stages do not fit in shared memory");
      pl->d_nab = nab;
      pl->d_abytes = 0;
      pl->d_nstage = ns;
      pl->d_stage = st;
      pl->d_smem = ns * st + extra;
    } else {
      const uint32_t st = NC * 128u + 16384u;
      const uint32_t extra = ctl + slack;
      int ns = static_cast<int>((kSmemMax - extra) / st);
      if (ns > 8) ns = 8;
      if (ns < 2) return fail(MAPL_ERR_UNSUPPORTED, "decompress stages do not fit in shared memory");
      pl->d_nab = 0;
      pl->d_abytes = 0;
      pl->d_nstage = ns;
      pl->d_stage = st;
      pl->d_smem = ns * st + extra;
    }
  }
  return MAPL_OK;
}

mapl_status build_plan_maps(mapl_plan_s* pl) {
  const mapl_config& c = pl->cfg;
  const uint32_t nrow = c.r > 256 ? 256u : static_cast<uint32_t>(c.r);
  const uint64_t NC = pl->d_nc;
  if (!make_tmap(&pl->tmAt, pl->p.At, c.d, c.r, 64, nrow))
    return fail(MAPL_ERR_CUDA, "cuTensorMapEncodeTiled failed (A^T)");
  if (!make_tmap(&pl->tmMt, pl->p.Mts, c.r, static_cast<uint64_t>(kNumSplit) * c.r, 64, nrow))
    return fail(MAPL_ERR_CUDA, "cuTensorMapEncodeTiled failed (M splits)");
  // [A | P'^T] (d x 2r): the persistent decompress loads two K-blocks per
  // stage as one 3-D box {64, NC, 2}; the streamed one loads 2-D boxes
  if (!(pl->d_stream ? make_tmap(&pl->tmB, pl->p.Bcat, 2 * c.r, c.d, 64, static_cast<uint32_t>(NC))
                     : make_tmap_atoms(&pl->tmB, pl->p.Bcat, 2 * c.r, c.d,
                                       static_cast<uint32_t>(NC), 2)))
    return fail(MAPL_ERR_CUDA, "cuTensorMapEncodeTiled failed ([A | P'^T])");
  if (pl->vq) {
    // one book per load, rows of gd bf16 in the swizzle that matches the row
    // width (64 B: SWIZZLE_64B, 32 B: SWIZZLE_32B)
    const CUtensorMapSwizzle swz =
        pl->gd == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
    if (!make_tmap(&pl->tmC, pl->p.Cb, static_cast<uint64_t>(pl->gd),
                   static_cast<uint64_t>(c.R) * c.G * c.K, static_cast<uint32_t>(pl->gd),
                   static_cast<uint32_t>(c.K), swz))
      return fail(MAPL_ERR_CUDA, "cuTensorMapEncodeTiled failed (codebooks)");
    // norm rows: 16 bf16 (32 bytes) per code, one book per load
    if (!make_tmap(&pl->tmH, pl->p.Hs, 16, static_cast<uint64_t>(c.R) * c.G * c.K, 16,
                   static_cast<uint32_t>(c.K), CU_TENSOR_MAP_SWIZZLE_32B))
      return fail(MAPL_ERR_CUDA, "cuTensorMapEncodeTiled failed (norm rows)");
  } else {
    pl->tmC = pl->tmAt;   // unused
    pl->tmH = pl->tmAt;   // unused
  }
  return MAPL_OK;
}

mapl_status check_device(const mapl_plan_s* pl) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != pl->device)
    return fail(MAPL_ERR_INVALID_ARG, "current device %d differs from the plan's device %d", dev,
                pl->device);
  return MAPL_OK;
}

}  // namespace

extern "C" {

int32_t mapl_version(void) { return 100; }

const char* mapl_last_error(void) { return g_last_error.c_str(); }

mapl_status mapl_payload_bytes(const mapl_config* cfg, int64_t* bytes_per_token) {
  mapl_status st = validate(cfg);
  if (st != MAPL_OK) return st;
  if (!bytes_per_token) return fail(MAPL_ERR_INVALID_ARG, "bytes_per_token is NULL");
  if (cfg->G > 0)
    *bytes_per_token = static_cast<int64_t>(cfg->R) * cfg->G;
  else
    *bytes_per_token = cfg->r * static_cast<int64_t>(elt_size(*cfg));
  return MAPL_OK;
}

static mapl_status plan_M(mapl_plan pl, cudaStream_t stream);

mapl_status mapl_plan_create(mapl_plan* out, const mapl_config* cfg, const void* A,
                             const void* P_send, const void* P_recv, const void* codebooks,
                             cudaStream_t stream) {
  if (!out) return fail(MAPL_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  mapl_status st = validate(cfg);
  if (st != MAPL_OK) return st;
  const bool vq = cfg->G > 0;
  if (!A || !P_send || !P_recv) return fail(MAPL_ERR_INVALID_ARG, "A, P_send, P_recv must be non-NULL");
  if (vq && !codebooks) return fail(MAPL_ERR_INVALID_ARG, "codebooks must be non-NULL with VQ");
  if (!vq && codebooks) return fail(MAPL_ERR_INVALID_ARG, "codebooks given without VQ");
  if (!aligned16(A) || !aligned16(P_send) || !aligned16(P_recv) || (codebooks && !aligned16(codebooks)))
    return fail(MAPL_ERR_INVALID_ARG, "parameter pointers must be 16-byte aligned");

  mapl_plan_s* pl = new mapl_plan_s();
  pl->cfg = *cfg;
  pl->vq = vq;
  pl->tc = cfg->dtype == MAPL_BF16;
  pl->gd = vq ? static_cast<int>(cfg->r / cfg->G) : 0;
  pl->re = static_cast<int>(cfg->r);
  cudaError_t e = cudaGetDevice(&pl->device);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&pl->num_sms, cudaDevAttrMultiProcessorCount, pl->device);
  if (e != cudaSuccess) {
    delete pl;
    return cuda_fail(e, "cudaGetDevice");
  }
  const int64_t d = cfg->d, r = cfg->r;
  const int64_t nb = vq ? static_cast<int64_t>(cfg->R) * cfg->G : 0;
  const int64_t ncode = nb * (vq ? cfg->K : 0);
  // one pool for every plan-owned buffer
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off += up256(bytes); return o; };
  size_t oAt = 0, oMts = 0, oBcat = 0, oCb = 0, oHs = 0, oA32 = 0, oAt32 = 0, oM32 = 0,
         oC32 = 0;
  const size_t oPs = take(d * r * elt_size(*cfg));
  const size_t oPr = take(d * r * elt_size(*cfg));
  if (pl->tc) {
    oAt = take(d * r * 2);
    oM32 = take(r * r * 4);
    oMts = take(static_cast<size_t>(kNumSplit) * r * r * 2);
    oBcat = take(d * 2 * r * 2);
    if (vq) oCb = take(ncode * pl->gd * 2);
    if (vq) oHs = take(ncode * 16 * 2);
  } else {
    oA32 = take(d * r * 4);
    oAt32 = take(d * r * 4);
    oM32 = take(r * r * 4);
    if (vq) oC32 = take(ncode * pl->gd * 4);
  }
  const size_t ocn = take((ncode > 0 ? ncode : 1) * 4);
  const size_t ocm = take((nb > 0 ? nb : 1) * 4);
  const size_t oerr = take(8);   // the error word, then the codebook-update counter
  void* pool = nullptr;
  e = cudaMalloc(&pool, off);
  if (e != cudaSuccess) {
    delete pl;
    return cuda_fail(e, "cudaMalloc(plan)");
  }
  char* b = reinterpret_cast<char*>(pool);
  PlanDevice& p = pl->p;
  p.pool = pool;
  if (pl->tc) {
    p.At = reinterpret_cast<__nv_bfloat16*>(b + oAt);
    p.M32 = reinterpret_cast<float*>(b + oM32);
    p.Mts = reinterpret_cast<__nv_bfloat16*>(b + oMts);
    p.Bcat = reinterpret_cast<__nv_bfloat16*>(b + oBcat);
    if (vq) p.Cb = reinterpret_cast<__nv_bfloat16*>(b + oCb);
    if (vq) p.Hs = reinterpret_cast<__nv_bfloat16*>(b + oHs);
  } else {
    p.A32 = reinterpret_cast<float*>(b + oA32);
    p.At32 = reinterpret_cast<float*>(b + oAt32);
    p.M32 = reinterpret_cast<float*>(b + oM32);
    p.Pr32 = reinterpret_cast<float*>(b + oPr);
    if (vq) p.C32 = reinterpret_cast<float*>(b + oC32);
  }
  p.Ps = b + oPs;
  p.Pr = b + oPr;
  p.cnorm = reinterpret_cast<float*>(b + ocn);
  p.cmax = reinterpret_cast<float*>(b + ocm);
  p.err = reinterpret_cast<int*>(b + oerr);
  p.upd_ctr = reinterpret_cast<unsigned int*>(b + oerr + 4);

  e = cudaMemsetAsync(p.err, 0, 8, stream);   // the error word and the update counter
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(p.Ps, P_send, d * r * elt_size(*cfg), cudaMemcpyDeviceToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(p.Pr, P_recv, d * r * elt_size(*cfg), cudaMemcpyDeviceToDevice, stream);
  if (e == cudaSuccess)
    e = pl->tc ? launch_prep_bf16(*cfg, A, p.Ps, p.Pr, codebooks, p, false, stream)
               : launch_prep_f32(*cfg, A, p.Ps, p.Pr, codebooks, p, false, stream);
  if (e == cudaSuccess && pl->tc) {
    st = plan_M(pl, stream);
    if (st != MAPL_OK) {
      cudaStreamSynchronize(stream);
      if (pl->blas) cublasDestroy(pl->blas);
      cudaFree(pool);
      delete pl;
      return st;
    }
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    if (pl->blas) cublasDestroy(pl->blas);
    cudaFree(pool);
    delete pl;
    return cuda_fail(e, "plan preparation");
  }
  if (pl->tc) {
    st = geometry(pl);
    if (st == MAPL_OK) st = build_plan_maps(pl);
    if (st != MAPL_OK) {
      if (pl->blas) cublasDestroy(pl->blas);
      cudaFree(pool);
      delete pl;
      return st;
    }
  }
  *out = pl;
  return MAPL_OK;
}

static mapl_status blas_on(mapl_plan pl, cudaStream_t stream) {
  if (!pl->blas && cublasCreate(&pl->blas) != CUBLAS_STATUS_SUCCESS) {
    pl->blas = nullptr;
    return fail(MAPL_ERR_CUDA, "cublasCreate failed");
  }
  if (cublasSetStream(pl->blas, stream) != CUBLAS_STATUS_SUCCESS)
    return fail(MAPL_ERR_CUDA, "cublasSetStream failed");
  return MAPL_OK;
}

// bf16 plan: M = P_send A (r x r) from the plan's A^T and P_send copies, a
// plain GEMM (cuBLAS, bf16 products exact, fp32 accumulation: M to about
// 2^-24 relative, far inside what the fold's three bf16 terms carry into Z),
// then -M^T split into the three bf16 terms of the anchor fold.
static mapl_status plan_M(mapl_plan pl, cudaStream_t stream) {
  mapl_status st = blas_on(pl, stream);
  if (st != MAPL_OK) return st;
  const mapl_config& c = pl->cfg;
  const int r = static_cast<int>(c.r), d = static_cast<int>(c.d);
  // column-major: M^T (r x r) = A^T P_send^T; the row-major A^T (r x d) is
  // the column-major d x r A, read transposed; the row-major P_send (r x d)
  // is the column-major d x r P_send^T.  The column-major M^T is the
  // row-major M.
  const float one = 1.f, zero = 0.f;
  const cublasStatus_t bs =
      cublasGemmEx(pl->blas, CUBLAS_OP_T, CUBLAS_OP_N, r, r, d, &one, pl->p.At, CUDA_R_16BF, d,
                   pl->p.Ps, CUDA_R_16BF, d, &zero, pl->p.M32, CUDA_R_32F, r, CUBLAS_COMPUTE_32F,
                   CUBLAS_GEMM_DEFAULT);
  if (bs != CUBLAS_STATUS_SUCCESS) return fail(MAPL_ERR_CUDA, "cuBLAS GEMM failed (%d)", (int)bs);
  const cudaError_t e = launch_split_negMt(pl->p.M32, r, pl->p.Mts, stream);
  if (e != cudaSuccess) return cuda_fail(e, "anchor fold operand");
  return MAPL_OK;
}

// T = E_emb A (cuBLAS, bf16 in, fp32 out) split into the [hi|mid|lo] table.
static mapl_status embedding_table(mapl_plan pl, cudaStream_t stream) {
  const mapl_config& c = pl->cfg;
  mapl_status bst = blas_on(pl, stream);
  if (bst != MAPL_OK) return bst;
  // column-major: T^T (r x V) = A^T * E_emb^T, with the plan's row-major
  // A^T (r x d) read as the column-major d x r matrix A and transposed
  const float one = 1.f, zero = 0.f;
  const cublasStatus_t bs = cublasGemmEx(
      pl->blas, CUBLAS_OP_T, CUBLAS_OP_N, static_cast<int>(c.r), static_cast<int>(c.V),
      static_cast<int>(c.d), &one, pl->p.At, CUDA_R_16BF, static_cast<int>(c.d), pl->E_emb,
      CUDA_R_16BF, static_cast<int>(c.d), &zero, pl->emb_T, CUDA_R_32F, static_cast<int>(c.r),
      CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
  if (bs != CUBLAS_STATUS_SUCCESS) return fail(MAPL_ERR_CUDA, "cuBLAS GEMM failed (%d)", (int)bs);
  const cudaError_t e = launch_split3(pl->emb_T, static_cast<size_t>(c.V), static_cast<int>(c.r),
                                      pl->emb_tab, stream);
  if (e != cudaSuccess) return cuda_fail(e, "embedding anchor table");
  return MAPL_OK;
}

mapl_status mapl_plan_set_embedding_anchor(mapl_plan pl, const void* E_emb, cudaStream_t stream) {
  if (!pl || !E_emb) return fail(MAPL_ERR_INVALID_ARG, "NULL argument");
  if (!pl->tc) return fail(MAPL_ERR_UNSUPPORTED, "the embedding anchor needs a bf16 plan");
  if (!aligned16(E_emb)) return fail(MAPL_ERR_INVALID_ARG, "E_emb must be 16-byte aligned");
  if (3 * pl->cfg.r > 512)
    return fail(MAPL_ERR_UNSUPPORTED, "the embedding anchor needs r <= 170 (3r table columns)");
  mapl_status st = check_device(pl);
  if (st != MAPL_OK) return st;
  const mapl_config& c = pl->cfg;
  const size_t r = static_cast<size_t>(c.r), V = static_cast<size_t>(c.V);
  const size_t oT = 0, oTab = up256(V * r * 4), oM = oTab + up256(V * 3 * r * 2);
  cudaError_t e;
  if (!pl->emb_pool) {
    e = cudaMalloc(&pl->emb_pool, oM + up256(r * 3 * r * 2));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(embedding anchor)");
  }
  char* b = static_cast<char*>(pl->emb_pool);
  pl->emb_T = reinterpret_cast<float*>(b + oT);
  pl->emb_tab = reinterpret_cast<__nv_bfloat16*>(b + oTab);
  __nv_bfloat16* M = reinterpret_cast<__nv_bfloat16*>(b + oM);
  e = launch_neg_identity3(static_cast<int>(r), M, stream);
  if (e != cudaSuccess) return cuda_fail(e, "embedding anchor operand");
  const uint32_t nrow = c.r > 256 ? 256u : static_cast<uint32_t>(c.r);
  if (!make_tmap(&pl->tmMt_emb, M, 3 * r, r, 64, nrow))
    return fail(MAPL_ERR_CUDA, "cuTensorMapEncodeTiled failed (-[I;I;I])");
  pl->E_emb = E_emb;
  st = embedding_table(pl, stream);
  if (st != MAPL_OK) {
    pl->E_emb = nullptr;
    return st;
  }
  pl->re = static_cast<int>(3 * r);
  pl->nsplit = 1;
  return MAPL_OK;
}

mapl_status mapl_plan_update_A(mapl_plan pl, const void* A, cudaStream_t stream) {
  if (!pl || !A) return fail(MAPL_ERR_INVALID_ARG, "plan and A must be non-NULL");
  if (!aligned16(A)) return fail(MAPL_ERR_INVALID_ARG, "A must be 16-byte aligned");
  mapl_status st = check_device(pl);
  if (st != MAPL_OK) return st;
  cudaError_t e = pl->tc ? launch_prep_bf16(pl->cfg, A, pl->p.Ps, pl->p.Pr, nullptr, pl->p, true, stream)
                         : launch_prep_f32(pl->cfg, A, pl->p.Ps, pl->p.Pr, nullptr, pl->p, true, stream);
  if (e != cudaSuccess) return cuda_fail(e, "update_A");
  if (pl->tc) {
    const mapl_status st = plan_M(pl, stream);
    if (st != MAPL_OK) return st;
  }
  if (pl->E_emb) return embedding_table(pl, stream);
  return MAPL_OK;
}

mapl_status mapl_plan_update_codes(mapl_plan pl, const int32_t* ids, int32_t count,
                                   const void* codes, cudaStream_t stream) {
  if (!pl) return fail(MAPL_ERR_INVALID_ARG, "plan is NULL");
  if (!pl->vq) return fail(MAPL_ERR_INVALID_ARG, "the plan has no codebooks");
  if (count < 0) return fail(MAPL_ERR_INVALID_ARG, "count must be >= 0");
  if (count == 0) return MAPL_OK;
  if (!ids || !codes) return fail(MAPL_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(codes) || (reinterpret_cast<uintptr_t>(ids) & 3u))
    return fail(MAPL_ERR_INVALID_ARG, "codes must be 16-byte aligned (ids 4-byte)");
  mapl_status st = check_device(pl);
  if (st != MAPL_OK) return st;
  cudaError_t e = launch_update_codes(pl->cfg, ids, count, codes, pl->p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "update_codes");
  return MAPL_OK;
}

namespace {

// splitmix64 (Steele, Lea, Flood 2014; Vigna's reference constants): the
// counter-based generator both ends of a boundary run to agree on the subset.
uint64_t splitmix64(uint64_t& x) {
  x += 0x9E3779B97F4A7C15ull;
  uint64_t z = x;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

}  // namespace

mapl_status mapl_stream_subset(int64_t total, int64_t per_batch, uint64_t seed, int64_t step,
                               int32_t* ids, int32_t* count) {
  if (total < 1 || total > 0x7fffffffLL) return fail(MAPL_ERR_INVALID_ARG, "total must be in [1, 2^31)");
  if (per_batch < 1 || per_batch > total)
    return fail(MAPL_ERR_INVALID_ARG, "per_batch must be in [1, total]");
  if (step < 0 || !ids || !count)
    return fail(MAPL_ERR_INVALID_ARG, "step must be >= 0, ids and count non-NULL");
  // epoch e = step / nsub is a fresh permutation of [0, total) (Fisher-Yates
  // driven by splitmix64 seeded with seed and e); step takes its
  // (step % nsub)-th block of per_batch codes (the last block is shorter)
  const int64_t nsub = (total + per_batch - 1) / per_batch;
  const int64_t epoch = step / nsub, blk = step % nsub;
  std::vector<int32_t> perm(static_cast<size_t>(total));
  for (int64_t i = 0; i < total; ++i) perm[static_cast<size_t>(i)] = static_cast<int32_t>(i);
  uint64_t state = seed ^ (0xD1B54A32D192ED03ull * static_cast<uint64_t>(epoch + 1));
  for (int64_t i = total - 1; i > 0; --i) {
    const uint64_t j = splitmix64(state) % static_cast<uint64_t>(i + 1);
    std::swap(perm[static_cast<size_t>(i)], perm[static_cast<size_t>(j)]);
  }
  const int64_t b = blk * per_batch, e = std::min(total, b + per_batch);
  for (int64_t i = b; i < e; ++i) ids[i - b] = perm[static_cast<size_t>(i)];
  *count = static_cast<int32_t>(e - b);
  return MAPL_OK;
}

void mapl_plan_destroy(mapl_plan pl) {
  if (!pl) return;
  if (pl->blas) cublasDestroy(pl->blas);
  if (pl->emb_pool) cudaFree(pl->emb_pool);
  if (pl->gpool) cudaFree(pl->gpool);
  if (pl->p.pool) cudaFree(pl->p.pool);
  delete pl;
}

// grad_books: quantise with the plan's gradient codebooks (MCVQ of the
// backward gradient) instead of the forward ones.
static mapl_status compress_common(mapl_plan pl, const void* X, const int32_t* tids, int64_t N,
                                   const void* E, void* out, int mode, cudaStream_t stream,
                                   bool anchor = true, bool grad_books = false) {
  if (!pl) return fail(MAPL_ERR_INVALID_ARG, "plan is NULL");
  const bool own_table = pl->E_emb != nullptr;   // E_send is not read
  if (!X || !out || (anchor && (!tids || (!E && !own_table))))
    return fail(MAPL_ERR_INVALID_ARG, "NULL tensor pointer");
  if (N < 1 || N > 0x7fffffffLL) return fail(MAPL_ERR_INVALID_ARG, "N must be in [1, 2^31)");
  if (!aligned16(X) || !aligned16(out) ||
      (anchor && ((!own_table && !aligned16(E)) || (reinterpret_cast<uintptr_t>(tids) & 3u))))
    return fail(MAPL_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned (tids 4-byte)");
  mapl_status st = check_device(pl);
  if (st != MAPL_OK) return st;
  const mapl_config& c = pl->cfg;
  cudaError_t e;
  if (!anchor && !pl->tc)
    return fail(MAPL_ERR_UNSUPPORTED, "gradient calls need a bf16 (tensor-core) plan");
  if (!pl->tc) {
    e = launch_compress_f32(c, pl->p, reinterpret_cast<const float*>(X), tids, N,
                            reinterpret_cast<const float*>(E), out, mode, stream);
    if (e != cudaSuccess) return cuda_fail(e, "compress launch");
    return MAPL_OK;
  }
  CUtensorMap tmX, tmE;
  if (!make_tmap(&tmX, X, c.d, static_cast<uint64_t>(N), 64, kTile))
    return fail(MAPL_ERR_CUDA, "cuTensorMapEncodeTiled failed (X)");
  const bool emb = anchor && pl->E_emb != nullptr;
  if (emb) E = pl->emb_tab;   // first-boundary anchor: the plan's own table
  if (anchor) {
    if (!make_tmap(&tmE, E, static_cast<uint64_t>(pl->re), static_cast<uint64_t>(c.V), 64, 1))
      return fail(MAPL_ERR_CUDA, "cuTensorMapEncodeTiled failed (E)");
  } else {
    tmE = tmX;   // unused
  }
  CompressArgs a{};
  a.tids = tids;
  a.E = reinterpret_cast<const __nv_bfloat16*>(E);
  a.re = pl->re;
  a.nsplit = pl->nsplit;
  a.Cb = grad_books ? pl->Cb_g : pl->p.Cb;
  a.cnorm = grad_books ? pl->cnorm_g : pl->p.cnorm;
  a.cmax = grad_books ? pl->cmax_g : pl->p.cmax;
  a.out = out;
  a.err = pl->p.err;
  a.N = static_cast<int>(N);
  a.d = static_cast<int>(c.d);
  a.r = static_cast<int>(c.r);
  a.V = static_cast<int>(c.V);
  a.G = c.G;
  a.R = c.R;
  a.K = c.K;
  a.gd = pl->gd;
  a.mode = mode;
  a.anchor = anchor ? 1 : 0;
  a.nstage = pl->c_nstage;
  a.stage_bytes = pl->c_stage;
  a.timeout_ns = pl->timeout_ns;
  if (pl->c_pipe) {
    // one contiguous range of about N / grid rows per CTA, at least 64 rows
    a.nstage = pl->p_nx;
    a.stage_bytes = 16384u;
    a.nbstage = pl->p_nb;
    a.bstage_bytes = pl->p_bstage;
    a.ncb = pl->p_ncb;
    a.cstage_bytes = pl->p_cstage;
    const int64_t want = (N + 63) / 64;
    const int grid = static_cast<int>(want < pl->num_sms ? want : pl->num_sms);
    e = launch_compress_pipe(tmX, pl->tmAt, emb ? pl->tmMt_emb : pl->tmMt,
                             grad_books ? pl->tmC_g : pl->tmC, grad_books ? pl->tmH_g : pl->tmH,
                             tmE, a, pl->p_smem, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e, "compress launch");
    return MAPL_OK;
  }
  const int ntiles = static_cast<int>((N + kTile - 1) / kTile);
  const int grid = ntiles < pl->num_sms ? ntiles : pl->num_sms;
  e = launch_compress_tc(tmX, pl->tmAt, emb ? pl->tmMt_emb : pl->tmMt,
                         grad_books ? pl->tmC_g : pl->tmC, tmE, a, pl->c_smem, grid, stream);
  if (e != cudaSuccess) return cuda_fail(e, "compress launch");
  return MAPL_OK;
}

mapl_status mapl_compress(mapl_plan pl, const void* X, const int32_t* tids, int64_t N,
                          const void* E_send, void* payload, cudaStream_t stream) {
  if (!pl) return fail(MAPL_ERR_INVALID_ARG, "plan is NULL");
  const int mode = pl->vq ? kModeVQ : (pl->tc ? kModeZ16 : kModeZ32);
  return compress_common(pl, X, tids, N, E_send, payload, mode, stream);
}

mapl_status mapl_compress_z32(mapl_plan pl, const void* X, const int32_t* tids, int64_t N,
                              const void* E_send, float* Z, cudaStream_t stream) {
  return compress_common(pl, X, tids, N, E_send, Z, kModeZ32, stream);
}

// anchor == false: the E' term is left out (backward pass, dX = gZ A^T) and
// the payload is a bf16 N x r tensor, or (grad_books) VQ indices into the
// plan's gradient codebooks.
static mapl_status decompress_common(mapl_plan pl, const void* payload, const int32_t* tids,
                                     int64_t N, const void* E_recv, void* X_hat,
                                     cudaStream_t stream, bool anchor, bool grad_books = false) {
  if (!pl) return fail(MAPL_ERR_INVALID_ARG, "plan is NULL");
  // first-boundary anchor: X_hat = Z_hat A^T + E_emb[tids], E_recv not read
  const bool emb = anchor && pl->E_emb != nullptr;
  if (!payload || !X_hat || (anchor && (!tids || (!E_recv && !emb))))
    return fail(MAPL_ERR_INVALID_ARG, "NULL tensor pointer");
  if (N < 1 || N > 0x7fffffffLL) return fail(MAPL_ERR_INVALID_ARG, "N must be in [1, 2^31)");
  if (!aligned16(payload) || !aligned16(X_hat) ||
      (anchor && ((!emb && !aligned16(E_recv)) || (reinterpret_cast<uintptr_t>(tids) & 3u))))
    return fail(MAPL_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned (tids 4-byte)");
  mapl_status st = check_device(pl);
  if (st != MAPL_OK) return st;
  const mapl_config& c = pl->cfg;
  cudaError_t e;
  if (!anchor && !pl->tc)
    return fail(MAPL_ERR_UNSUPPORTED, "gradient calls need a bf16 (tensor-core) plan");
  const bool vq = anchor ? pl->vq : grad_books;
  if (!pl->tc) {
    e = launch_decompress_f32(c, pl->p, payload, tids, N, reinterpret_cast<const float*>(E_recv),
                              reinterpret_cast<float*>(X_hat), stream);
    if (e != cudaSuccess) return cuda_fail(e, "decompress launch");
    return MAPL_OK;
  }
  CUtensorMap tmZ;
  if (!vq) {
    if (!make_tmap(&tmZ, payload, c.r, static_cast<uint64_t>(N), 64, kTile))
      return fail(MAPL_ERR_CUDA, "cuTensorMapEncodeTiled failed (Z)");
  } else {
    tmZ = pl->tmB;   // unused
  }
  DecompressArgs a{};
  a.tids = tids;
  a.E = reinterpret_cast<const __nv_bfloat16*>(E_recv);
  a.Cb = grad_books ? pl->Cb_g : pl->p.Cb;
  a.idx = vq ? reinterpret_cast<const uint8_t*>(payload) : nullptr;
  a.Zp = vq ? nullptr : reinterpret_cast<const __nv_bfloat16*>(payload);
  a.Xh = reinterpret_cast<__nv_bfloat16*>(X_hat);
  a.err = pl->p.err;
  a.N = static_cast<int>(N);
  a.d = static_cast<int>(c.d);
  a.r = static_cast<int>(c.r);
  a.V = static_cast<int>(c.V);
  a.G = c.G;
  a.R = c.R;
  a.K = c.K;
  a.gd = pl->gd;
  a.vq = vq ? 1 : 0;
  a.anchor = anchor && !emb ? 1 : 0;
  a.Eadd = emb ? reinterpret_cast<const __nv_bfloat16*>(pl->E_emb) : nullptr;
  a.a_stream = pl->d_stream ? 1 : 0;
  a.nc = static_cast<int>(pl->d_nc);
  a.nab = pl->d_nab;
  a.nstage = pl->d_nstage;
  a.stage_bytes = pl->d_stage;
  a.a_bytes = pl->d_abytes;
  a.timeout_ns = pl->timeout_ns;
  const int ntiles = static_cast<int>((N + kTile - 1) / kTile);
  if (pl->d_nab > 0) {
    CUtensorMap tmXh;
    if (!make_tmap(&tmXh, X_hat, c.d, static_cast<uint64_t>(N), 64, 32))
      return fail(MAPL_ERR_CUDA, "cuTensorMapEncodeTiled failed (X_hat)");
    // one contiguous range of 32-row blocks per CTA
    const int64_t nb32 = (N + 31) / 32;
    const int grid = static_cast<int>(nb32 < pl->num_sms ? nb32 : pl->num_sms);
    e = launch_decompress_pt(pl->tmB, tmXh, a, pl->d_smem, grid, stream);
  } else {
    if (emb) return fail(MAPL_ERR_UNSUPPORTED, "the embedding anchor needs the persistent decompress");
    e = launch_decompress_tc(pl->tmB, tmZ, a, pl->d_smem, ntiles, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "decompress launch");
  return MAPL_OK;
}

mapl_status mapl_decompress(mapl_plan pl, const void* payload, const int32_t* tids, int64_t N,
                            const void* E_recv, void* X_hat, cudaStream_t stream) {
  return decompress_common(pl, payload, tids, N, E_recv, X_hat, stream, true);
}

// ------------------------------------------------------------ backward pass
mapl_status mapl_grad_compress(mapl_plan pl, const void* gX_hat, int64_t N, void* gZ,
                               cudaStream_t stream) {
  return compress_common(pl, gX_hat, nullptr, N, nullptr, gZ, kModeZ16, stream, false);
}

mapl_status mapl_grad_decompress(mapl_plan pl, const void* gZ, int64_t N, void* gX,
                                 cudaStream_t stream) {
  return decompress_common(pl, gZ, nullptr, N, nullptr, gX, stream, false);
}

mapl_status mapl_plan_set_grad_codebooks(mapl_plan pl, const void* codebooks, cudaStream_t stream) {
  if (!pl || !codebooks) return fail(MAPL_ERR_INVALID_ARG, "NULL argument");
  if (!pl->vq || !pl->tc)
    return fail(MAPL_ERR_UNSUPPORTED, "gradient codebooks need a bf16 VQ plan");
  if (!aligned16(codebooks)) return fail(MAPL_ERR_INVALID_ARG, "codebooks must be 16-byte aligned");
  mapl_status st = check_device(pl);
  if (st != MAPL_OK) return st;
  const mapl_config& c = pl->cfg;
  const size_t nb = static_cast<size_t>(c.R) * c.G, ncode = nb * c.K;
  const size_t ohs = up256(ncode * pl->gd * sizeof(__nv_bfloat16));
  const size_t ocn = ohs + up256(ncode * 16 * sizeof(__nv_bfloat16));
  const size_t ocm = ocn + up256(ncode * sizeof(float));
  if (!pl->gpool) {
    cudaError_t e = cudaMalloc(&pl->gpool, ocm + up256(nb * sizeof(float)));
    if (e != cudaSuccess) {
      pl->gpool = nullptr;
      return cuda_fail(e, "cudaMalloc(gradient codebooks)");
    }
    char* b = static_cast<char*>(pl->gpool);
    pl->Cb_g = reinterpret_cast<__nv_bfloat16*>(b);
    pl->Hs_g = reinterpret_cast<__nv_bfloat16*>(b + ohs);
    pl->cnorm_g = reinterpret_cast<float*>(b + ocn);
    pl->cmax_g = reinterpret_cast<float*>(b + ocm);
    const CUtensorMapSwizzle swz =
        pl->gd == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
    if (!make_tmap(&pl->tmC_g, pl->Cb_g, static_cast<uint64_t>(pl->gd), ncode,
                   static_cast<uint32_t>(pl->gd), static_cast<uint32_t>(c.K), swz) ||
        !make_tmap(&pl->tmH_g, pl->Hs_g, 16, ncode, 16, static_cast<uint32_t>(c.K),
                   CU_TENSOR_MAP_SWIZZLE_32B))
      return fail(MAPL_ERR_CUDA, "cuTensorMapEncodeTiled failed (gradient codebooks)");
  }
  const cudaError_t e = launch_prep_books_bf16(c, codebooks, pl->Cb_g, pl->Hs_g, pl->cnorm_g,
                                               pl->cmax_g, stream);
  if (e != cudaSuccess) return cuda_fail(e, "gradient codebook prep");
  return MAPL_OK;
}

mapl_status mapl_grad_compress_vq(mapl_plan pl, const void* gX_hat, int64_t N, void* payload,
                                  cudaStream_t stream) {
  if (!pl) return fail(MAPL_ERR_INVALID_ARG, "plan is NULL");
  if (!pl->gpool) return fail(MAPL_ERR_INVALID_ARG, "no gradient codebooks (mapl_plan_set_grad_codebooks)");
  return compress_common(pl, gX_hat, nullptr, N, nullptr, payload, kModeVQ, stream, false, true);
}

mapl_status mapl_grad_decompress_vq(mapl_plan pl, const void* payload, int64_t N, void* gX,
                                    cudaStream_t stream) {
  if (!pl) return fail(MAPL_ERR_INVALID_ARG, "plan is NULL");
  if (!pl->gpool) return fail(MAPL_ERR_INVALID_ARG, "no gradient codebooks (mapl_plan_set_grad_codebooks)");
  return decompress_common(pl, payload, nullptr, N, nullptr, gX, stream, false, true);
}

namespace {

// Token splits, tiles and K block of the projector gradient for N tokens.
struct GradGeom {
  int nX, nE, S, W, nM, kb, nstage;
  bool fold;
  uint32_t smem;
  size_t ws_bar, ws_partials, ws_fold, ws_T, ws_total;
};

// Column tiles of W = 256 (128 when r = 512, so that the r / 128 M blocks of
// 128 x W fp32 accumulators fit TMEM's 512 columns), 32-token blocks, as many
// ring stages as shared memory holds, and S token splits per tile so that
// the grid is at most one CTA per SM.
GradGeom grad_geom(const mapl_plan_s* pl, int64_t N) {
  const mapl_config& c = pl->cfg;
  GradGeom g{};
  const bool emb = pl->E_emb != nullptr;
  g.fold = !emb && c.r <= 128;
  g.W = c.r <= 256 ? 256 : 128;
  g.nM = static_cast<int>((c.r + 127) / 128);
  g.nX = static_cast<int>((c.d + g.W - 1) / g.W);
  g.nE = emb ? g.nX : (g.fold ? 0 : static_cast<int>((c.r + g.W - 1) / g.W));
  g.kb = 32;
  const uint32_t st = grad_stage_bytes(static_cast<int>(c.r), g.W, g.kb);
  int ns = static_cast<int>((kSmemMax - 2048u - grad_ctl_bytes() - grad_fring_bytes(g.kb)) / st);
  if (ns > kGradMaxStages) ns = kGradMaxStages;
  g.nstage = ns;
  g.smem = ns * st + grad_fring_bytes(g.kb) + 1024u + grad_ctl_bytes() + 64u;
  const int64_t nkb = (N + g.kb - 1) / g.kb;
  int S = pl->num_sms / (g.nX + g.nE);
  if (S < 1) S = 1;
  if (S > nkb) S = static_cast<int>(nkb);
  g.S = S;
  g.ws_bar = 256;
  g.ws_partials = up256(static_cast<size_t>(g.nX + g.nE) * S * g.W * c.r * sizeof(float));
  g.ws_fold = g.fold ? up256(static_cast<size_t>(g.nX) * S * c.r * c.r * sizeof(float)) : 0;
  g.ws_T = up256(static_cast<size_t>(c.r) * c.r * sizeof(float));
  g.ws_total = g.ws_bar + g.ws_partials + g.ws_fold + g.ws_T;
  return g;
}

}  // namespace

mapl_status mapl_grad_workspace_size(mapl_plan pl, int64_t N, size_t* bytes) {
  if (!pl || !bytes) return fail(MAPL_ERR_INVALID_ARG, "NULL argument");
  if (N < 1 || N > 0x7fffffffLL) return fail(MAPL_ERR_INVALID_ARG, "N must be in [1, 2^31)");
  if (!pl->tc) return fail(MAPL_ERR_UNSUPPORTED, "gradient calls need a bf16 (tensor-core) plan");
  *bytes = grad_geom(pl, N).ws_total;
  return MAPL_OK;
}

mapl_status mapl_grad_A(mapl_plan pl, const void* X, const int32_t* tids, const void* E_send,
                        const void* gZ, const void* gX_hat, const void* Z, int64_t N, float* dA,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!pl) return fail(MAPL_ERR_INVALID_ARG, "plan is NULL");
  const bool emb = pl->E_emb != nullptr;   // first-boundary anchor: E_send is not read
  if (!X || !tids || (!E_send && !emb) || !gZ || !gX_hat || !Z || !dA || !workspace)
    return fail(MAPL_ERR_INVALID_ARG, "NULL pointer argument");
  if (N < 1 || N > 0x7fffffffLL) return fail(MAPL_ERR_INVALID_ARG, "N must be in [1, 2^31)");
  if (!pl->tc) return fail(MAPL_ERR_UNSUPPORTED, "gradient calls need a bf16 (tensor-core) plan");
  if (!aligned16(X) || !aligned16(gZ) || !aligned16(gX_hat) || !aligned16(Z) || !aligned16(dA) ||
      (!emb && !aligned16(E_send)) || (reinterpret_cast<uintptr_t>(tids) & 3u))
    return fail(MAPL_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned (tids 4-byte)");
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(MAPL_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  mapl_status st = check_device(pl);
  if (st != MAPL_OK) return st;
  const mapl_config& c = pl->cfg;
  const GradGeom g = grad_geom(pl, N);
  if (workspace_bytes < g.ws_total)
    return fail(MAPL_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes,
                g.ws_total);
  // MN-major slabs: boxes of 64 elements x kb tokens x the slab's 64-element
  // atoms (W / 64 of X and dL/dX_hat, 2 per 128 rows of r of gZ and Z); the
  // anchor table of an E tile by four-row gathers of one 64-element segment
  const uint32_t kb = static_cast<uint32_t>(g.kb);
  const uint32_t nB = static_cast<uint32_t>(g.W / 64), nA = static_cast<uint32_t>(2 * g.nM);
  CUtensorMap tmX, tmGX, tmGZ, tmZ, tmE;
  if (!make_tmap_atoms(&tmX, X, c.d, static_cast<uint64_t>(N), kb, nB) ||
      !make_tmap_atoms(&tmGX, gX_hat, c.d, static_cast<uint64_t>(N), kb, nB) ||
      !make_tmap_atoms(&tmGZ, gZ, c.r, static_cast<uint64_t>(N), kb, nA) ||
      !make_tmap_atoms(&tmZ, Z, c.r, static_cast<uint64_t>(N), kb, nA))
    return fail(MAPL_ERR_CUDA, "cuTensorMapEncodeTiled failed (gradient operands)");
  const void* table = emb ? pl->E_emb : E_send;
  const uint64_t tcols = emb ? static_cast<uint64_t>(c.d) : static_cast<uint64_t>(c.r);
  if (!make_tmap(&tmE, table, tcols, static_cast<uint64_t>(c.V), 64, 1))
    return fail(MAPL_ERR_CUDA, "cuTensorMapEncodeTiled failed (anchor table)");
  char* wsb = static_cast<char*>(workspace);
  GradArgs a{};
  a.tids = tids;
  a.E = static_cast<const __nv_bfloat16*>(E_send);
  a.P = reinterpret_cast<const __nv_bfloat16*>(pl->p.Ps);
  a.err = pl->p.err;
  a.bar = reinterpret_cast<unsigned int*>(wsb);
  a.ws = reinterpret_cast<float*>(wsb + g.ws_bar);
  a.wsT = reinterpret_cast<float*>(wsb + g.ws_bar + g.ws_partials);
  a.T = reinterpret_cast<float*>(wsb + g.ws_bar + g.ws_partials + g.ws_fold);
  a.dA = dA;
  a.N = static_cast<int>(N);
  a.d = static_cast<int>(c.d);
  a.r = static_cast<int>(c.r);
  a.V = static_cast<int>(c.V);
  a.S = g.S;
  a.nX = g.nX;
  a.nE = g.nE;
  a.W = g.W;
  a.nM = g.nM;
  a.kb = g.kb;
  a.nstage = g.nstage;
  a.emb = emb ? 1 : 0;
  a.fold = g.fold ? 1 : 0;
  a.timeout_ns = pl->timeout_ns;
  const cudaError_t e =
      launch_grad_A(tmX, tmGX, tmGZ, tmZ, tmE, a, (g.nX + g.nE) * g.S, g.smem, stream);
  if (e != cudaSuccess) return cuda_fail(e, "gradient launch");
  return MAPL_OK;
}

// ---------------------------------------------------------- host buffers
namespace {

struct HostLayout {
  size_t x, tids, payload, total;
};

void payload_bytes_of(const mapl_config& c, int64_t* bytes) {
  *bytes = c.G > 0 ? static_cast<int64_t>(c.R) * c.G : c.r * static_cast<int64_t>(elt_size(c));
}

HostLayout host_layout(const mapl_plan_s* pl, int64_t N) {
  const mapl_config& c = pl->cfg;
  int64_t pbytes = 0;
  payload_bytes_of(c, &pbytes);
  HostLayout h{};
  h.x = 0;
  h.tids = h.x + up256(static_cast<size_t>(N) * c.d * elt_size(c));
  h.payload = h.tids + up256(static_cast<size_t>(N) * 4);
  h.total = h.payload + up256(static_cast<size_t>(N) * pbytes);
  return h;
}

mapl_status host_args(const mapl_plan_s* pl, int64_t N, const void* a, const void* b,
                      const void* c, void* ws, size_t ws_bytes, HostLayout* h) {
  if (!pl) return fail(MAPL_ERR_INVALID_ARG, "plan is NULL");
  if (!a || !b || !c || !ws) return fail(MAPL_ERR_INVALID_ARG, "NULL pointer");
  if (N < 1 || N > 0x7fffffffLL) return fail(MAPL_ERR_INVALID_ARG, "N must be in [1, 2^31)");
  if (reinterpret_cast<uintptr_t>(ws) & 255u)
    return fail(MAPL_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  *h = host_layout(pl, N);
  if (ws_bytes < h->total)
    return fail(MAPL_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", ws_bytes, h->total);
  return MAPL_OK;
}

}  // namespace

mapl_status mapl_host_workspace_size(mapl_plan pl, int64_t N, size_t* bytes) {
  if (!pl || !bytes) return fail(MAPL_ERR_INVALID_ARG, "NULL argument");
  if (N < 1 || N > 0x7fffffffLL) return fail(MAPL_ERR_INVALID_ARG, "N must be in [1, 2^31)");
  *bytes = host_layout(pl, N).total;
  return MAPL_OK;
}

mapl_status mapl_compress_host(mapl_plan pl, const void* X, const int32_t* tids, int64_t N,
                               const void* E_send, void* payload, void* ws, size_t ws_bytes,
                               cudaStream_t stream) {
  HostLayout h{};
  mapl_status st = host_args(pl, N, X, tids, payload, ws, ws_bytes, &h);
  if (st != MAPL_OK) return st;
  const mapl_config& c = pl->cfg;
  int64_t pbytes = 0;
  payload_bytes_of(c, &pbytes);
  char* w = reinterpret_cast<char*>(ws);
  cudaError_t e = cudaMemcpyAsync(w + h.x, X, static_cast<size_t>(N) * c.d * elt_size(c),
                                  cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(w + h.tids, tids, static_cast<size_t>(N) * 4, cudaMemcpyHostToDevice,
                        stream);
  if (e != cudaSuccess) return cuda_fail(e, "host -> device copy");
  st = mapl_compress(pl, w + h.x, reinterpret_cast<const int32_t*>(w + h.tids), N, E_send,
                     w + h.payload, stream);
  if (st != MAPL_OK) return st;
  e = cudaMemcpyAsync(payload, w + h.payload, static_cast<size_t>(N) * pbytes,
                      cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return cuda_fail(e, "device -> host copy");
  return MAPL_OK;
}

mapl_status mapl_decompress_host(mapl_plan pl, const void* payload, const int32_t* tids,
                                 int64_t N, const void* E_recv, void* X_hat, void* ws,
                                 size_t ws_bytes, cudaStream_t stream) {
  HostLayout h{};
  mapl_status st = host_args(pl, N, payload, tids, X_hat, ws, ws_bytes, &h);
  if (st != MAPL_OK) return st;
  const mapl_config& c = pl->cfg;
  int64_t pbytes = 0;
  payload_bytes_of(c, &pbytes);
  char* w = reinterpret_cast<char*>(ws);
  cudaError_t e = cudaMemcpyAsync(w + h.payload, payload, static_cast<size_t>(N) * pbytes,
                                  cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(w + h.tids, tids, static_cast<size_t>(N) * 4, cudaMemcpyHostToDevice,
                        stream);
  if (e != cudaSuccess) return cuda_fail(e, "host -> device copy");
  st = mapl_decompress(pl, w + h.payload, reinterpret_cast<const int32_t*>(w + h.tids), N, E_recv,
                       w + h.x, stream);
  if (st != MAPL_OK) return st;
  e = cudaMemcpyAsync(X_hat, w + h.x, static_cast<size_t>(N) * c.d * elt_size(c),
                      cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return cuda_fail(e, "device -> host copy");
  return MAPL_OK;
}

mapl_status mapl_store_probe(void* dst, size_t bytes, int32_t mode, cudaStream_t stream) {
  if (!dst) return fail(MAPL_ERR_INVALID_ARG, "dst is NULL");
  if (!aligned16(dst) || bytes % 16 != 0)
    return fail(MAPL_ERR_INVALID_ARG, "dst must be 16-byte aligned and bytes a multiple of 16");
  if (mode < 0 || mode > 2) return fail(MAPL_ERR_INVALID_ARG, "mode must be 0, 1 or 2");
  if (bytes == 0) return MAPL_OK;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = launch_store_probe(dst, bytes, mode, sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "store probe");
  return MAPL_OK;
}

mapl_status mapl_selftest_bounded_wait(mapl_plan pl, int64_t budget_ns, int64_t* waited_ns,
                                       cudaStream_t stream) {
  if (!pl || !waited_ns) return fail(MAPL_ERR_INVALID_ARG, "NULL argument");
  if (budget_ns < 1000 || budget_ns > 2000000000LL)
    return fail(MAPL_ERR_INVALID_ARG, "budget_ns must be in [1 us, 2 s]");
  mapl_status st = check_device(pl);
  if (st != MAPL_OK) return st;
  unsigned long long* d = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&d), sizeof(*d), stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync");
  unsigned long long h = 0;
  e = launch_wait_selftest(static_cast<uint64_t>(budget_ns), pl->p.err, d, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&h, d, sizeof(h), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  cudaFreeAsync(d, stream);
  if (e != cudaSuccess) return cuda_fail(e, "bounded-wait self-test");
  *waited_ns = static_cast<int64_t>(h);
  return MAPL_OK;
}

mapl_status mapl_check(mapl_plan pl, cudaStream_t stream) {
  if (!pl) return fail(MAPL_ERR_INVALID_ARG, "plan is NULL");
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int w = 0;
  e = cudaMemcpy(&w, pl->p.err, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  if (w) {
    e = cudaMemset(pl->p.err, 0, 4);
    if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  }
  if (w & kErrTimeout) return fail(MAPL_ERR_TIMEOUT, "an in-kernel wait gave up");
  if (w & kErrBadToken) return fail(MAPL_ERR_BAD_TOKEN, "a token id was outside [0, V)");
  if (w & kErrBadIndex) return fail(MAPL_ERR_INVALID_ARG, "a VQ index in the payload was >= K");
  return MAPL_OK;
}

mapl_status mapl_spel_workspace_size(int64_t d, int64_t r, int32_t batch, size_t* bytes) {
  if (!bytes) return fail(MAPL_ERR_INVALID_ARG, "bytes is NULL");
  if (d < 4 || r < 4 || d % 4 || r % 4 || r > d || batch < 1 || d > (1 << 20))
    return fail(MAPL_ERR_INVALID_ARG, "need 4 | d, 4 | r, r <= d, batch >= 1");
  *bytes = spel_workspace_bytes(d, r, batch);
  return MAPL_OK;
}

mapl_status mapl_spel_step(float* A, const float* G, float* m, int64_t d, int64_t r,
                           int32_t batch, float lr, float beta, const float* coeffs,
                           int32_t n_lmo, int32_t n_retr, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  if (!A || !G || !m || !coeffs || !workspace)
    return fail(MAPL_ERR_INVALID_ARG, "NULL pointer argument");
  size_t need = 0;
  mapl_status st = mapl_spel_workspace_size(d, r, batch, &need);
  if (st != MAPL_OK) return st;
  if (workspace_bytes < need)
    return fail(MAPL_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
  if (n_lmo < 0 || n_retr < 0 || n_lmo + n_retr < 1 || n_lmo + n_retr > 32)
    return fail(MAPL_ERR_INVALID_ARG, "need 1 <= n_lmo + n_retr <= 32");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) || !aligned16(A) || !aligned16(G) || !aligned16(m))
    return fail(MAPL_ERR_INVALID_ARG, "workspace must be 256-byte, tensors 16-byte aligned");
  if (!(beta >= 0.f && beta < 1.f)) return fail(MAPL_ERR_INVALID_ARG, "beta must be in [0, 1)");
  cudaError_t e = launch_spel(A, G, m, static_cast<int>(d), static_cast<int>(r), batch, lr, beta,
                              coeffs, n_lmo, n_retr, workspace, stream);
  if (e != cudaSuccess) return cuda_fail(e, "spel launch");
  return MAPL_OK;
}

mapl_status mapl_spel_step_refresh(float* A, const float* G, float* m, int64_t d, int64_t r,
                                   int32_t batch, float lr, float beta, const float* coeffs,
                                   int32_t n_lmo, int32_t n_retr, const mapl_plan* plans,
                                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!plans) return fail(MAPL_ERR_INVALID_ARG, "plans is NULL");
  if (batch < 1 || batch > kMaxRefresh)
    return fail(MAPL_ERR_UNSUPPORTED, "the fused plan refresh takes 1 to %d boundaries", kMaxRefresh);
  RefreshTable rt{};
  rt.n = batch;
  for (int b = 0; b < batch; ++b) {
    mapl_plan pl = plans[b];
    if (!pl) continue;
    if (!pl->tc) return fail(MAPL_ERR_UNSUPPORTED, "plan %d: the fused refresh needs a bf16 plan", b);
    if (pl->cfg.d != d || pl->cfg.r != r)
      return fail(MAPL_ERR_INVALID_ARG, "plan %d has (d, r) = (%lld, %lld), the step (%lld, %lld)",
                  b, static_cast<long long>(pl->cfg.d), static_cast<long long>(pl->cfg.r),
                  static_cast<long long>(d), static_cast<long long>(r));
    for (int q = 0; q < b; ++q)
      if (plans[q] == pl) return fail(MAPL_ERR_INVALID_ARG, "plan %d appears twice", b);
    mapl_status st = check_device(pl);
    if (st != MAPL_OK) return st;
    rt.At[b] = pl->p.At;
    rt.Bcat[b] = pl->p.Bcat;
  }
  if (!A || !G || !m || !coeffs || !workspace)
    return fail(MAPL_ERR_INVALID_ARG, "NULL pointer argument");
  size_t need = 0;
  mapl_status st = mapl_spel_workspace_size(d, r, batch, &need);
  if (st != MAPL_OK) return st;
  if (workspace_bytes < need)
    return fail(MAPL_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
  if (n_lmo < 0 || n_retr < 0 || n_lmo + n_retr < 1 || n_lmo + n_retr > 32)
    return fail(MAPL_ERR_INVALID_ARG, "need 1 <= n_lmo + n_retr <= 32");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) || !aligned16(A) || !aligned16(G) || !aligned16(m))
    return fail(MAPL_ERR_INVALID_ARG, "workspace must be 256-byte, tensors 16-byte aligned");
  if (!(beta >= 0.f && beta < 1.f)) return fail(MAPL_ERR_INVALID_ARG, "beta must be in [0, 1)");
  cudaError_t e = launch_spel(A, G, m, static_cast<int>(d), static_cast<int>(r), batch, lr, beta,
                              coeffs, n_lmo, n_retr, workspace, stream, &rt);
  if (e != cudaSuccess) return cuda_fail(e, "spel launch");
  for (int b = 0; b < batch; ++b) {
    if (!plans[b]) continue;
    st = plan_M(plans[b], stream);   // M = P_send bf16(A) from the A^T just written
    if (st == MAPL_OK && plans[b]->E_emb) st = embedding_table(plans[b], stream);
    if (st != MAPL_OK) return st;
  }
  return MAPL_OK;
}

mapl_status mapl_spel_step_static(float* A, const float* G, float* m, int64_t d, int64_t r,
                                  int32_t batch, float lr, float beta, const float* coeffs,
                                  int32_t n_lmo, int32_t n_retr, cudaStream_t stream) {
  if (!A || !G || !m || !coeffs) return fail(MAPL_ERR_INVALID_ARG, "NULL pointer argument");
  size_t need = 0;
  mapl_status st = mapl_spel_workspace_size(d, r, batch, &need);
  if (st != MAPL_OK) return st;
  if (need > kSpelStaticScratchBytes)
    return fail(MAPL_ERR_UNSUPPORTED,
                "mapl_spel_step_static: (d=%lld, r=%lld, batch=%d) needs %zu bytes of scratch, "
                "more than the fixed %zu; use mapl_spel_step with a caller workspace",
                static_cast<long long>(d), static_cast<long long>(r), batch, need,
                kSpelStaticScratchBytes);
  if (n_lmo < 0 || n_retr < 0 || n_lmo + n_retr < 1 || n_lmo + n_retr > 32)
    return fail(MAPL_ERR_INVALID_ARG, "need 1 <= n_lmo + n_retr <= 32");
  if (!aligned16(A) || !aligned16(G) || !aligned16(m))
    return fail(MAPL_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (!(beta >= 0.f && beta < 1.f)) return fail(MAPL_ERR_INVALID_ARG, "beta must be in [0, 1)");
  void* scratch = nullptr;
  cudaError_t e = spel_static_scratch(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static SPEL scratch)");
  e = launch_spel(A, G, m, static_cast<int>(d), static_cast<int>(r), batch, lr, beta, coeffs,
                  n_lmo, n_retr, scratch, stream);
  if (e != cudaSuccess) return cuda_fail(e, "spel launch");
  return MAPL_OK;
}

}  // extern "C"
