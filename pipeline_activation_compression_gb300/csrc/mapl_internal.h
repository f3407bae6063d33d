// mapl_internal.h -- plan layout and kernel launchers shared by the host API
// (mapl_api.cu) and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mapl.h"

namespace mapl {

constexpr int kTile = 128;          // tokens per CTA tile (MMA M)
constexpr int kNumSplit = 3;        // bf16 terms of -M in the folded anchor product
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s per bounded wait

// device error word bits (mapl_check maps them to mapl_status)
constexpr int kErrBadToken = 1;
constexpr int kErrTimeout = 2;
constexpr int kErrBadIndex = 4;

// Compress kernel modes.
enum CompressMode { kModeZ16 = 0, kModeVQ = 1, kModeZ32 = 2 };

struct PlanDevice {
  // bf16 tensor-core operands
  __nv_bfloat16* At = nullptr;      // r x d     A^T (K-major B operand of X A)
  __nv_bfloat16* Mts = nullptr;     // S x r x r -M^T split into S bf16 terms
  __nv_bfloat16* Bcat = nullptr;    // d x 2r    [A | P_recv^T] (K-major B of decompress)
  __nv_bfloat16* Cb = nullptr;      // R x G x K x gd codebooks (B operand of the distance
                                    // MMA, decode lookups)
  __nv_bfloat16* Hs = nullptr;      // R x G x K x 16 norm rows [h_hi, h_mid, h_lo, 0 ...]:
                                    // ||c||^2 / 2 as three bf16 terms (B operand of the
                                    // distance MMA's norm product)
  // fp32 CUDA-core path
  float* A32 = nullptr;             // d x r
  float* At32 = nullptr;            // r x d     A^T
  float* M32 = nullptr;             // r x r     M = P_send A (both paths)
  float* Pr32 = nullptr;            // r x d     P_recv
  float* C32 = nullptr;             // R x G x K x gd
  // both
  void* Ps = nullptr;               // r x d     copy of P_send (plan dtype)
  void* Pr = nullptr;               // r x d     copy of P_recv (plan dtype)
  float* cnorm = nullptr;           // R x G x K  ||c||^2 (fp32 of the exact value)
  float* cmax = nullptr;            // R x G      max_k ||c_k|| (rounded up)
  int* err = nullptr;               // device error word (bits kErrBadToken, kErrTimeout)
  unsigned int* upd_ctr = nullptr;  // blocks of a codebook update done (0 between calls)
  void* pool = nullptr;             // single allocation holding everything above
};

struct CompressArgs {
  const int32_t* tids;
  const __nv_bfloat16* E;           // V x r
  const __nv_bfloat16* Cb;
  const float* cnorm;
  const float* cmax;
  void* out;
  int* err;
  int N, d, r, V, G, R, K, gd;
  int mode;
  int anchor;                       // 0: no anchor term (backward pass: gZ = dX_hat A)
  int re;                           // columns of the anchor table E (multiple of 64)
  int nsplit;                       // bf16 terms of -M (re x r) in the folded anchor
  int nstage;                       // X ring stages (pipelined kernel) / ring stages
  uint32_t stage_bytes;
  int nbstage;                      // pipelined kernel: B ring stages (A^T, -M^T blocks)
  uint32_t bstage_bytes;            //   r x 128 bytes
  int ncb;                          //   codebook ring stages (VQ)
  uint32_t cstage_bytes;            //   K x gd x 2 bytes of codes + K x 32 bytes of norm rows
  uint64_t timeout_ns;
};

struct DecompressArgs {
  const int32_t* tids;
  const __nv_bfloat16* E;           // V x r (receiver)
  const __nv_bfloat16* Cb;
  const uint8_t* idx;               // VQ payload (N x R x G) or null
  const __nv_bfloat16* Zp;          // bf16 payload Z_hat (N x r) when not VQ
  __nv_bfloat16* Xh;                // N x d
  int* err;
  int N, d, r, V, G, R, K, gd;
  int vq;
  int a_stream;                     // A operand streamed per stage (r > 256)
  int nc;                           // output columns per accumulator chunk
  int nab;                          // A operand buffers (persistent kernel)
  int anchor;                       // 0: no E' term (backward pass: dX = gZ A^T)
  const __nv_bfloat16* Eadd;        // V x d rows added to X_hat (first-boundary anchor) or null
  int nstage;
  uint32_t stage_bytes;
  uint32_t a_bytes;                 // resident A operand bytes (0 when streamed)
  uint64_t timeout_ns;
};

uint32_t compress_ctl_bytes();      // control block of the compress kernel
uint32_t compress_pipe_ctl_bytes(); // control block of the pipelined compress kernel
uint32_t compress_pipe_ones_bytes(); // its constant A tile of the norm product (VQ)
// Shapes the pipelined compress kernel handles: without VQ r <= 256; with
// VQ r in {64, 128}, group width 16 or 32, an even number of groups, K a
// multiple of 128.
bool compress_pipe_supported(int r, bool vq, int gd, int G, int K);
uint32_t decompress_ctl_bytes();    // control block of the decompress kernel
uint32_t decompress_pt_ctl_bytes(); // control block + drain staging of the persistent kernel

// ---- launchers (return cudaGetLastError() of the launch) -------------------
cudaError_t launch_prep_bf16(const mapl_config& c, const void* A, const void* Ps, const void* Pr,
                             const void* C, PlanDevice& p, bool A_only, cudaStream_t s);
cudaError_t launch_prep_f32(const mapl_config& c, const void* A, const void* Ps, const void* Pr,
                            const void* C, PlanDevice& p, bool A_only, cudaStream_t s);

// One warp waits (bounded) on an mbarrier nothing arrives on; sets the
// timeout bit of `err` when it gives up and writes the time waited.
cudaError_t launch_store_probe(void* dst, size_t bytes, int mode, int num_sms, cudaStream_t s);
cudaError_t launch_prep_books_bf16(const mapl_config& c, const void* C, __nv_bfloat16* Cb,
                                   __nv_bfloat16* Hs, float* cnorm, float* cmax, cudaStream_t s);
cudaError_t launch_wait_selftest(uint64_t budget_ns, int* err, unsigned long long* waited,
                                 cudaStream_t s);
cudaError_t launch_update_codes(const mapl_config& c, const int32_t* ids, int count,
                                const void* codes, PlanDevice& p, cudaStream_t s);

cudaError_t launch_compress_tc(const CUtensorMap& tmX, const CUtensorMap& tmAt,
                               const CUtensorMap& tmMt, const CUtensorMap& tmC,
                               const CUtensorMap& tmE, const CompressArgs& a,
                               uint32_t smem_bytes, int grid, cudaStream_t s);
cudaError_t launch_compress_pipe(const CUtensorMap& tmX, const CUtensorMap& tmAt,
                                 const CUtensorMap& tmMt, const CUtensorMap& tmC,
                                 const CUtensorMap& tmH, const CUtensorMap& tmE,
                                 const CompressArgs& a, uint32_t smem_bytes, int grid,
                                 cudaStream_t s);
cudaError_t launch_decompress_pt(const CUtensorMap& tmB, const CUtensorMap& tmXh,
                                 const DecompressArgs& a, uint32_t smem_bytes, int grid,
                                 cudaStream_t s);
// Projector gradient on the tensor cores (kernels_grad_tc.cu).  Output
// tiles: nX of 128 rows of d (X^T gZ + gXh^T Z) and nE of 128 rows of the
// anchor table's columns (E[tids]^T gZ), each split into S token ranges of
// whole K blocks of kb tokens; partials in ws, (nX + nE) x S x 128 x r fp32.
struct GradArgs {
  const int32_t* tids;
  const __nv_bfloat16* E;           // E_send (V x r), factored anchor
  const __nv_bfloat16* P;           // P_send (r x d), factored anchor
  int* err;
  unsigned int* bar;                // grid-barrier counter, zeroed before the launch
  float* ws;                        // column-tile partials, (nX + nE) x S x W x r
  float* wsT;                       // folded anchor partials, nX x S x r x r (fold only)
  float* T;                         // E[tids]^T gZ, r x r (factored anchor)
  float* dA;
  int N, d, r, V;
  int S, nX, nE, W, nM, kb, nstage;
  int emb;                          // first-boundary anchor: E tiles over d, subtracted
  int fold;                         // factored anchor folded into the X tiles (r <= 128)
  uint64_t timeout_ns;
};
constexpr int kGradMaxStages = 8;
uint32_t grad_stage_bytes(int r, int W, int kb);
uint32_t grad_fring_bytes(int kb);   // the folded-gather ring, whole
uint32_t grad_ctl_bytes();
cudaError_t launch_grad_A(const CUtensorMap& tmX, const CUtensorMap& tmGX, const CUtensorMap& tmGZ,
                          const CUtensorMap& tmZ, const CUtensorMap& tmE, const GradArgs& a,
                          int grid, uint32_t smem, cudaStream_t s);
// First-boundary anchor: T (V x r fp32) -> [hi | mid | lo] bf16 (V x 3r), and
// the r x 3r operand -[I; I; I]^T.
cudaError_t launch_split3(const float* T, size_t V, int r, __nv_bfloat16* Tb, cudaStream_t s);
cudaError_t launch_neg_identity3(int r, __nv_bfloat16* M, cudaStream_t s);
cudaError_t launch_decompress_tc(const CUtensorMap& tmB, const CUtensorMap& tmZ,
                                 const DecompressArgs& a, uint32_t smem_bytes, int grid,
                                 cudaStream_t s);

cudaError_t launch_compress_f32(const mapl_config& c, const PlanDevice& p, const float* X,
                                const int32_t* tids, int64_t N, const float* E, void* out,
                                int mode, cudaStream_t s);
cudaError_t launch_decompress_f32(const mapl_config& c, const PlanDevice& p, const void* in,
                                  const int32_t* tids, int64_t N, const float* E, float* Xh,
                                  cudaStream_t s);

size_t spel_workspace_bytes(int64_t d, int64_t r, int32_t batch);

// Size of the fixed device scratch behind mapl_spel_step_static (16 MiB).
constexpr size_t kSpelStaticScratchBytes = static_cast<size_t>(16) << 20;
// Device address of that scratch on the current device (cudaGetSymbolAddress
// on every call, never cached).
cudaError_t spel_static_scratch(void** out);
// Plan operands written by a SPEL step's last retraction product from the
// new fp32 A (rounded to bf16), per boundary of the batch; boundaries with
// At == nullptr are skipped.  M is formed afterwards by the host API.
constexpr int kMaxRefresh = 16;
struct RefreshTable {
  int n;
  __nv_bfloat16* At[kMaxRefresh];     // r x d
  __nv_bfloat16* Bcat[kMaxRefresh];   // d x 2r, columns [0, r) written
};
cudaError_t launch_spel(float* A, const float* G, float* m, int d, int r, int batch, float lr,
                        float beta, const float* coeffs, int n_lmo, int n_retr, void* ws,
                        cudaStream_t s, const RefreshTable* rt = nullptr);
// Mts = -M^T in kNumSplit bf16 terms from the fp32 r x r M of a bf16 plan.
// Batched fp32 product on the tensor cores (3-term bf16 split, six term
// products, fp32 accumulation): C[z] + ks * sS = opA[z] * opB[z]^T over split
// ks of K.  An operand holds `rows x K` values, element (row, k) at
// p[row * ld + k], or at p[k * ld + row] when rows_contig.  Needs M, N
// multiples of 128 and K a multiple of 64 * ksplit (gemm3_supported).
struct Gemm3Operand {
  const float* p;
  long ld;
  long batch_stride;
  int rows_contig;
};
bool gemm3_supported(int M, int N, int K, int ksplit);
cudaError_t launch_gemm3(const Gemm3Operand& a, const Gemm3Operand& b, float* C, long ldc,
                         long sC, long sS, int M, int N, int K, int batch, int ksplit,
                         cudaStream_t s);

cudaError_t launch_split_negMt(const float* M, int r, __nv_bfloat16* Mts, cudaStream_t s);

}  // namespace mapl
