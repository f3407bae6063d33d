/*
 * mapl.h -- C ABI of the MAPL boundary codec for one GB300 (sm_103a).
 *
 * MAPL ("Learned Subspace Compression for Communication-Efficient Pipeline
 * Parallelism") compresses the activation that crosses a pipeline-stage
 * boundary.  This library implements its per-micro-batch hot path and its
 * projector update:
 *
 *   compress    (§3.2 eq. (1), folded):  Z = X A - E_send[tids] (P_send A)
 *               optionally followed by multi-codebook residual VQ (§3.5)
 *   decompress  (§3.2 eq. (2)):          X_hat = Z_hat A^T + E_recv[tids] P_recv
 *               computed as one contraction [Z_hat | E_recv[tids]] [A^T ; P_recv]
 *   SPEL step   (§3.3 eqs. (4)-(7)):     tangent projection, heavy-ball
 *               momentum, PolarExpress LMO direction, PolarExpress retraction
 *
 * Conventions for every call below:
 *  - Every tensor pointer is a DEVICE pointer, row-major, contiguous, with a
 *    16-byte aligned base.  The caller owns all tensors; the library never
 *    frees or keeps them beyond the call, except where a plan copies a
 *    parameter (mapl_plan_create / mapl_plan_update_A).
 *  - Element type of X, A, P, E, codebooks, Z and X_hat is the plan's dtype:
 *    MAPL_BF16 (2-byte bfloat16 bit patterns) or MAPL_F32 (float).
 *    Token ids are int32; VQ indices are uint8.
 *  - Work is enqueued asynchronously on `stream` (0 = legacy default stream).
 *    The return value reports argument and launch errors only.  Errors that
 *    depend on data (a token id outside [0, V), an internal wait that gave up)
 *    are recorded in the plan's device error word and reported by mapl_check;
 *    the affected output rows are written as zeros.  No kernel traps.
 *  - Functions are thread-safe for distinct plans.  mapl_last_error() returns
 *    the message of the calling thread's most recent failure.
 */
#ifndef MAPL_H_
#define MAPL_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MAPL_OK = 0,
  MAPL_ERR_INVALID_ARG = 1,   /* null pointer, bad size or layout          */
  MAPL_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels handle */
  MAPL_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed         */
  MAPL_ERR_BAD_TOKEN = 4,     /* a token id was outside [0, V)             */
  MAPL_ERR_TIMEOUT = 5        /* a bounded in-kernel wait gave up          */
} mapl_status;

typedef enum { MAPL_F32 = 0, MAPL_BF16 = 1 } mapl_dtype;

/*
 * Boundary configuration (§3.2, §3.5, App. E.4).
 *   d  activation width, r  projection rank (St(d, r)), V  vocabulary size.
 *   G  VQ groups (gd = r / G dims each), R  residual rounds, K  codes per
 *   group and round.  G = R = K = 0 disables VQ: the payload is Z itself.
 * Limits: d % 64 == 0, r % 16 == 0, r <= 512, 1 <= V.  With VQ: G divides r,
 * 1 <= R <= 8, 1 <= K <= 256 (uint8 indices).  The bf16 tensor-core path
 * needs r % 64 == 0 and, with VQ, r <= 256, gd in {16, 32} and K % 64 == 0.
 * MAPL_F32 runs on CUDA cores in fp32 (any sizes within the limits above).
 */
typedef struct {
  int64_t d, r, V;
  int32_t G, R, K;
  int32_t dtype;   /* mapl_dtype */
  int32_t flags;   /* reserved, must be 0 */
} mapl_config;

typedef struct mapl_plan_s* mapl_plan;

/*
 * Create a plan for one boundary p.  Copies and re-lays-out the parameters:
 *   A          d x r   projector A_p in St(d, r)                (§3.2)
 *   P_send     r x d   sender's frozen anchor projector P_p      (eq. (3))
 *   P_recv     r x d   receiver's anchor projector P_{p+1}       (eq. (2))
 *   codebooks  R x G x K x gd  C[rho][g][k][:] (NULL without VQ) (§3.5)
 * and precomputes M = P_send A (r x r; bf16 plans: a cuBLAS GEMM with fp32
 * accumulation, fp32 plans: compensated fp32 sums), the operand
 * layouts of the kernels and the codebook norms.  The plan owns that device
 * memory; mapl_plan_destroy frees it.  Blocks until the copies are done.
 * Errors: INVALID_ARG (sizes, null), UNSUPPORTED, CUDA.
 */
mapl_status mapl_plan_create(mapl_plan* out, const mapl_config* cfg, const void* A,
                             const void* P_send, const void* P_recv,
                             const void* codebooks, cudaStream_t stream);

/* Replace A (d x r, plan dtype) after a projector update and refresh M and
 * the operand layouts (§3.3: A_p changes every optimizer step).  bf16 plans
 * form M with a cuBLAS GEMM on `stream` (the plan's handle is made at plan
 * creation, so the call can be captured in a CUDA graph).  Async. */
mapl_status mapl_plan_update_A(mapl_plan plan, const void* A, cudaStream_t stream);

/*
 * First-boundary anchor (Fig. 2 of the MAPL page: at the boundary after the
 * first stage the anchor is the original token embedding itself).  After
 * this call the plan's calls use
 *   compress    Z     = (X - E_emb[tids]) A
 *   decompress  X_hat = Z_hat A^T + E_emb[tids]
 *   grad_A      dA    = (X - E_emb[tids])^T gZ + gX_hat^T Z
 * and ignore their E_send / E_recv arguments (they may be NULL); P_send and
 * P_recv are no longer used.
 *   E_emb  V x d bf16, device, 16-byte aligned.  The plan keeps the POINTER
 *          (not a copy): the caller keeps E_emb alive and unchanged while the
 *          plan is used, and calls this again after changing it.
 * The compress fold E_emb[tids] A is read from a V x r table T = E_emb A that
 * the plan computes here and again in every mapl_plan_update_A (cuBLAS,
 * fp32 accumulation), held as three bf16 terms T_hi + T_mid + T_lo so the
 * tensor-core fold keeps about 24 bits of T.  Plan memory grows by
 * V x r x 10 bytes.  bf16 plans only, r <= 170.  Async on `stream`.
 * Errors: INVALID_ARG (null, alignment), UNSUPPORTED (f32 plan, r too
 * large), CUDA.
 */
mapl_status mapl_plan_set_embedding_anchor(mapl_plan plan, const void* E_emb, cudaStream_t stream);

/* Bytes of payload per token: 2r (bf16 Z), 4r (f32 Z) or R*G (uint8 idx). */
mapl_status mapl_payload_bytes(const mapl_config* cfg, int64_t* bytes_per_token);

/*
 * Sender side, eq. (1) with the anchor folded through M = P_send A:
 *   X       N x d   boundary activation X^{b_p}
 *   tids    N       token ids (int32, must lie in [0, V))
 *   E_send  V x r   sender's anchor table E_p^small
 *   payload without VQ: Z, N x r (plan dtype, bf16 rounded to nearest even);
 *           with VQ: indices, N x R x G uint8, idx[n][rho][g] = nearest code of
 *           group g's residual in round rho (lowest index on exact ties).
 * With VQ, Z never leaves the chip.  N >= 1.  Async.
 */
mapl_status mapl_compress(mapl_plan plan, const void* X, const int32_t* tids, int64_t N,
                          const void* E_send, void* payload, cudaStream_t stream);

/*
 * Diagnostic form of mapl_compress: runs the same projection (same kernel,
 * same accumulation order) and writes the fp32 Z (N x r float) that the VQ
 * stage would quantise, instead of the payload.  Used to bound the distance
 * error of the VQ decision in tests.  Async.
 */
mapl_status mapl_compress_z32(mapl_plan plan, const void* X, const int32_t* tids, int64_t N,
                              const void* E_send, float* Z, cudaStream_t stream);

/*
 * Receiver side, eq. (2):
 *   payload N x r Z (plan dtype) or N x R x G uint8 indices (decoded as
 *           Z_hat[n][g-block] = sum_rho C[rho][g][idx[n][rho][g]])
 *   tids    N, E_recv V x r (receiver's anchor table E_{p+1}^small)
 *   X_hat   N x d output (plan dtype; bf16 rounded to nearest even)
 * Async.
 */
mapl_status mapl_decompress(mapl_plan plan, const void* payload, const int32_t* tids,
                            int64_t N, const void* E_recv, void* X_hat, cudaStream_t stream);

/*
 * Streaming codebook synchronisation (MAPL §3.5, App. F): sender and receiver
 * keep identical codebooks by overwriting, each micro-batch, the same random
 * subset of codes with the sender's current values.  The pages give the
 * subset size as 1/K of the codes (§3.5), 1/5 per micro-batch (Table 8) and
 * "interval 5" (App. E.4); it is a parameter here.
 *
 * mapl_stream_subset (host only, no GPU): the subset for micro-batch `step`.
 *   The R*G*K codes (flat id = (rho*G + g)*K + k) are shuffled once per epoch
 *   of ceil(total / per_batch) steps (Fisher-Yates driven by splitmix64 seeded
 *   with `seed` and the epoch number), and step takes the epoch's
 *   (step mod steps-per-epoch)-th block of per_batch ids.  Writes *count ids
 *   (per_batch, or fewer for the last block of an epoch) to `ids`.  Both ends
 *   compute the same subset, so only the code values need to travel.
 * mapl_plan_update_codes: codes ids[i] (device int32) take the values
 *   codes[i * gd .. +gd) (device, plan dtype, 16-byte aligned); their ||c||^2 and every book's
 *   max ||c|| are refreshed.  An id outside [0, R*G*K) sets the error word
 *   (mapl_check reports MAPL_ERR_INVALID_ARG) and is skipped.  One launch
 *   (one block for up to 512 codes; for more, the last block to finish
 *   recomputes the maxima through a counter the plan keeps), so calls on
 *   the same plan must not overlap on the GPU, as with every call that
 *   writes the plan.  Async.
 */
mapl_status mapl_stream_subset(int64_t total, int64_t per_batch, uint64_t seed, int64_t step,
                               int32_t* ids, int32_t* count);

mapl_status mapl_plan_update_codes(mapl_plan plan, const int32_t* ids, int32_t count,
                                   const void* codes, cudaStream_t stream);

/*
 * Backward pass (MAPL §3.2: the gradient of the boundary activation is
 * routed through the same orthogonal projector A; §3.5: it is what the
 * gradient exchange compresses).  bf16 tensor-core plans only
 * (MAPL_ERR_UNSUPPORTED otherwise).  All pointers are device pointers.
 *
 * mapl_grad_compress   receiver side:  gZ = gX_hat A
 *   gX_hat  N x d  dL/dX_hat (bf16);  gZ  N x r  out (bf16, round to nearest
 *   even).  No anchor term: the anchor does not depend on X.
 * mapl_grad_decompress sender side:    gX = gZ A^T
 *   gZ  N x r (bf16);  gX  N x d out (bf16) = dL/dX through the codec.
 * mapl_grad_A          Euclidean gradient of A for SPEL:
 *   dA = X_res^T gZ + gX_hat^T Z,  X_res = X - E_send[tids] P_send
 *   X, gX_hat N x d; gZ, Z N x r (bf16; Z as the pipeline has it, e.g. the
 *   decoded payload); tids N; E_send V x r;  dA  d x r fp32 out.
 *   Computed as X^T gZ + gX_hat^T Z - P_send^T (E_send[tids]^T gZ) on the
 *   tensor cores (bf16 in, fp32 accumulation) in one cooperative launch
 *   (one CTA per SM; preceded by a 4-byte memset of the workspace's grid
 *   barrier), split over token ranges whose partial sums go to `workspace`
 *   and are then added in a fixed order, so the result is the same on every
 *   call (with an embedding-anchor plan, the last term is E_emb[tids]^T gZ
 *   and E_send may be NULL).  Token ids outside [0, V) contribute no anchor
 *   term and set MAPL_ERR_BAD_TOKEN in the plan's error word.
 *   workspace  device, 256-byte aligned, at least
 *              mapl_grad_workspace_size(plan, N) bytes, owned by the caller,
 *              not read before it is written; calls that overlap on the GPU
 *              need workspaces of their own.  The call allocates nothing.
 * mapl_grad_workspace_size  bytes of workspace mapl_grad_A needs for N tokens
 *   (about 30 MiB at d = 1024, r = 128 on 152 SMs).
 * Async on `stream`.
 */
mapl_status mapl_grad_compress(mapl_plan plan, const void* gX_hat, int64_t N, void* gZ,
                               cudaStream_t stream);

mapl_status mapl_grad_decompress(mapl_plan plan, const void* gZ, int64_t N, void* gX,
                                 cudaStream_t stream);

mapl_status mapl_grad_workspace_size(mapl_plan plan, int64_t N, size_t* bytes);

/*
 * MCVQ of backward gradients (MAPL §3.5: the multi-codebook quantiser
 * compresses both forward activations and backward gradients).  The
 * gradient has a distribution of its own, so it gets codebooks of its own:
 *   mapl_plan_set_grad_codebooks  R x G x K x gd bf16 codebooks (device,
 *     16-byte aligned), copied into the plan with their squared norms and
 *     per-book maxima; a later call replaces them.  The first call allocates
 *     their plan storage (R*G*K*(2 gd + 4) bytes).
 *   mapl_grad_compress_vq    gZ = dL/dX_hat A (no anchor term), quantised
 *     round by round with the gradient codebooks exactly as mapl_compress
 *     quantises Z (same kernel, same exact-nearest-code rule): payload
 *     N x (R*G) uint8, round-major then group.
 *   mapl_grad_decompress_vq  dL/dX = gZ_hat A^T, gZ_hat the sum over rounds of
 *     the payload's codes in the gradient codebooks; N x d bf16.
 * bf16 VQ plans only (UNSUPPORTED otherwise); the two codec calls return
 * INVALID_ARG until mapl_plan_set_grad_codebooks has been called.  Async.
 */
mapl_status mapl_plan_set_grad_codebooks(mapl_plan plan, const void* codebooks, cudaStream_t stream);

mapl_status mapl_grad_compress_vq(mapl_plan plan, const void* gX_hat, int64_t N, void* payload,
                                  cudaStream_t stream);

mapl_status mapl_grad_decompress_vq(mapl_plan plan, const void* payload, int64_t N, void* gX,
                                    cudaStream_t stream);

mapl_status mapl_grad_A(mapl_plan plan, const void* X, const int32_t* tids, const void* E_send,
                        const void* gZ, const void* gX_hat, const void* Z, int64_t N,
                        float* dA, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream);

/*
 * Host-buffer forms of mapl_compress / mapl_decompress, for callers whose
 * boundary activations live in host memory.  They are not part of the MAPL
 * method; they stage the host data through a caller-owned device workspace
 * on `stream`:
 *   mapl_compress_host:   X (N x d) and tids (N) are copied host -> device,
 *                         compressed, and the payload copied device -> host.
 *   mapl_decompress_host: payload and tids are copied host -> device,
 *                         decompressed, and X_hat (N x d) copied back.
 * X, tids, payload and X_hat are HOST pointers (pinned memory gives
 * asynchronous copies; pageable memory makes the copies synchronous);
 * E_send / E_recv stay DEVICE pointers (plan-lifetime tables).  workspace is
 * device memory of at least mapl_host_workspace_size(plan, N) bytes,
 * 256-byte aligned, owned by the caller and not shared by calls that may
 * overlap.  The output host buffer is written when the stream reaches the
 * end of the call.  Async; same errors as the device forms.
 */
mapl_status mapl_host_workspace_size(mapl_plan plan, int64_t N, size_t* bytes);

mapl_status mapl_compress_host(mapl_plan plan, const void* X, const int32_t* tids, int64_t N,
                               const void* E_send, void* payload, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream);

mapl_status mapl_decompress_host(mapl_plan plan, const void* payload, const int32_t* tids,
                                 int64_t N, const void* E_recv, void* X_hat, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream);

/*
 * Synchronise `stream`, then read and clear the plan's device error word.
 * Returns MAPL_OK, MAPL_ERR_BAD_TOKEN, MAPL_ERR_TIMEOUT, MAPL_ERR_CUDA, or
 * MAPL_ERR_INVALID_ARG when a decompressed payload held an index >= K (that
 * index was read as K - 1).
 */
mapl_status mapl_check(mapl_plan plan, cudaStream_t stream);

/*
 * Failure-detection self-test.  Every wait inside the codec kernels is
 * bounded: a kernel that gives up sets the timeout bit of the plan's error
 * word, unwinds and exits, so the context stays usable and mapl_check
 * returns MAPL_ERR_TIMEOUT.  This call runs that same bounded wait in a
 * one-warp kernel on an mbarrier that nothing arrives on, with a budget of
 * `budget_ns` (1 us .. 2 s), and blocks until it has given up.  The give-up
 * is recorded in the plan's error word exactly as a codec kernel records
 * it (so the next mapl_check returns MAPL_ERR_TIMEOUT); *waited_ns receives
 * the time the kernel waited.  Nothing else is launched or in flight.
 * Errors: INVALID_ARG, CUDA.
 */
mapl_status mapl_selftest_bounded_wait(mapl_plan plan, int64_t budget_ns, int64_t* waited_ns,
                                       cudaStream_t stream);

/*
 * Device write-rate probe (measurement only, no plan): writes `bytes` zero
 * bytes over `dst` (device, 16-byte aligned; bytes a multiple of 16) with
 * nothing read.  mode 0: 16-byte st.global from a grid-stride loop of four
 * 512-thread CTAs per SM; mode 1: the same with the streaming (evict-first)
 * hint; mode 2: bulk asynchronous copies (cp.async.bulk, the copy path of
 * the decompress kernel's TMA-store drain) of a zeroed 32 KB shared-memory
 * buffer, one CTA per SM over a contiguous range.  Timed on decompress's
 * own output buffers it gives the write ceiling decompress is held to.
 * Errors: INVALID_ARG, CUDA.
 */
mapl_status mapl_store_probe(void* dst, size_t bytes, int32_t mode, cudaStream_t stream);

void mapl_plan_destroy(mapl_plan plan);

/* Bytes of device workspace mapl_spel_step needs for (d, r, batch). */
mapl_status mapl_spel_workspace_size(int64_t d, int64_t r, int32_t batch, size_t* bytes);

/*
 * SPEL projector update (§3.3 eqs. (4)-(7), Algorithm 1 step 4) for `batch`
 * independent boundaries, fp32, in place:
 *   A   batch x d x r  projectors on St(d, r)      (updated)
 *   G   batch x d x r  Euclidean gradients dL/dA   (read)
 *   m   batch x d x r  momentum buffers            (updated)
 *   g_R = G - A sym(A^T G);  m = beta m + (1 - beta) g_R;
 *   D = PE(m / (||m||_F + 1e-7), LMO rows);  A = PE(A - lr D, retraction rows)
 * where PE applies Y <- Y (a I + b S + c S^2), S = Y^T Y, once per row.
 *   coeffs     HOST pointer, (n_lmo + n_retr) x 3 floats (a, b, c): the LMO
 *              rows first, then the retraction rows.  The pages give the
 *              iteration counts (5 / 7) but no coefficients.
 *   workspace  device scratch of at least mapl_spel_workspace_size bytes,
 *              owned by the caller, 256-byte aligned.
 * Requirements: r % 4 == 0, d % 4 == 0, r <= d, 1 <= n_lmo + n_retr <= 32.
 * Async.  The step's kernels are launched as programmatic dependent launches
 * (each waits for the stream's earlier work before it reads anything); a
 * kernel that the caller launches next with programmatic stream
 * serialization must itself wait (cudaGridDependencySynchronize) before it
 * reads A or m.  Ordinary launches, copies and events are ordered as usual.
 */
mapl_status mapl_spel_step(float* A, const float* G, float* m, int64_t d, int64_t r,
                           int32_t batch, float lr, float beta, const float* coeffs,
                           int32_t n_lmo, int32_t n_retr, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);

/*
 * mapl_spel_step_refresh -- mapl_spel_step, then the projector broadcast of
 * §3.3 ("the updated A_p is sent to the next stage after every optimizer
 * step") applied to the codec plans on this device: plans[b] (NULL to skip
 * boundary b) takes bf16(A[b]) (round to nearest even) as its projector, with
 * the same result as mapl_plan_update_A(plans[b], bf16(A[b])).  The final
 * retraction product writes the plans' A^T and [A | P_recv^T] operands in its
 * epilogue and one launch forms M = P_send A for every plan, so the refresh
 * adds no pass over A.  Embedding-anchor plans also recompute E_emb A.
 *   plans  HOST array of `batch` plan handles; bf16 plans with this (d, r),
 *          each at most once.  batch <= 16.
 * Other arguments and requirements as mapl_spel_step.  Async.
 * Errors: INVALID_ARG, UNSUPPORTED (f32 plan, batch > 16), CUDA.
 */
mapl_status mapl_spel_step_refresh(float* A, const float* G, float* m, int64_t d, int64_t r,
                                   int32_t batch, float lr, float beta, const float* coeffs,
                                   int32_t n_lmo, int32_t n_retr, const mapl_plan* plans,
                                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * mapl_spel_step_static -- the SPEL step above without a caller workspace.
 * The MAPL paper has no counterpart; this entry exists for callers that
 * cannot allocate device memory when they run the update: a framework whose
 * caching allocator has already reserved the device memory it is allowed to
 * use, a latency-bound loop that cannot afford cudaMalloc's implicit device
 * synchronisation, or a plugin interface whose fixed signature only passes
 * the tensors themselves.
 *
 * Same arguments and results as mapl_spel_step minus the workspace.  The
 * scratch is a fixed 16 MiB array in the library's device image, reserved on
 * every GPU that loads the library until the process exits;
 * mapl_spel_workspace_size(d, r, batch) must not exceed it (e.g. d = 1024,
 * r = 256, batch = 3 fits; d = 2048, r = 256, batch = 3 does not), otherwise
 * MAPL_ERR_UNSUPPORTED is returned and nothing runs.  The call allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine).
 *  - Every call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress), so the address stays right after a device
 *    reset.  The first call on a device also loads the library's device
 *    code there; make that first call before any stream capture.
 *  - All calls share the one array: calls whose work overlaps on the GPU
 *    (different streams, or several threads) race on it and must be
 *    serialised by the caller.  Nothing in the array needs to start at zero;
 *    each call overwrites what it reads.
 */
mapl_status mapl_spel_step_static(float* A, const float* G, float* m, int64_t d, int64_t r,
                                  int32_t batch, float lr, float beta, const float* coeffs,
                                  int32_t n_lmo, int32_t n_retr, cudaStream_t stream);

/* Message of the calling thread's last failed call ("" if none). */
const char* mapl_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t mapl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MAPL_H_ */
