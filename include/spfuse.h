/*
 * spfuse.h -- C ABI of libspfuse, the sequence-parallel (SP) region hot path
 * on one GB300 (sm_103a).
 *
 * The SP region is the per-token work between two tensor-parallel (TP)
 * regions: the reduce half of a reduce-scatter over the T row-parallel
 * partial outputs, dropout, the residual add and the next sub-layer's norm,
 * plus the backward of that chain and the sp2hp / hp2sp layout transforms.
 *
 * Sources (the pages this library follows):
 *  [MT3] MiniMind-tron ch.3 "Sequence Parallelism: layout and gradients"
 *  [MT4] MiniMind-tron ch.4 "Sequence Parallelism: memory bounds, async
 *        communication and recompute"
 *  [SPN] "Sequence Parallel" notes (cloudchewie), distributed training /
 *        parallelism
 *  [ATL] LLM Infra Atlas "03 · Sequence Parallelism: AG/RS replacing
 *        all-reduce"
 *
 * General conventions
 *  - Memory: every pointer argument is a DEVICE pointer (except the `partials`
 *    array itself, which is a host array of device pointers).  The caller owns
 *    all memory; the library never allocates, frees or synchronises.
 *  - Execution: every call enqueues its kernels on `stream` and returns
 *    without waiting.  Kernels are launched with programmatic dependent
 *    launch enabled; each kernel waits for the preceding work in the stream
 *    before it reads any input, so stream order is preserved.
 *  - Layout: activations are [S, B, H] row-major with the sequence as dim 0
 *    ([MT3] §3.2.4, [ATL] §3).  Sequence shard j of T is the contiguous row
 *    range [j*R, (j+1)*R) of the [S*B, H] view, R = (S/T)*B.
 *  - Validation: all arguments are checked before anything is launched; on
 *    error nothing is launched and the status says why.  A CUDA error at
 *    launch is reported as SP_ERR_CUDA.
 *  - Outputs must not alias inputs.  The library keeps no state between calls
 *    and is safe to call from several host threads.
 */
#ifndef SPFUSE_H
#define SPFUSE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* sp_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  SP_OK = 0,
  SP_ERR_INVALID_ARG = 1,     /* null pointer, bad p / eps / T / j */
  SP_ERR_SHAPE = 2,           /* S % T != 0, H not a multiple of the vector width, H too large */
  SP_ERR_ALIGN = 3,           /* a pointer is not aligned as required */
  SP_ERR_DTYPE = 4,           /* unknown dtype or norm */
  SP_ERR_WORKSPACE = 5,       /* workspace missing or smaller than required */
  SP_ERR_CUDA = 6,            /* a CUDA runtime call failed */
  SP_ERR_NOT_IMPLEMENTED = 7
} sp_status_t;

typedef enum { SP_F32 = 0, SP_BF16 = 1 } sp_dtype_t;
typedef enum { SP_RMSNORM = 0, SP_LAYERNORM = 1 } sp_norm_t;

/* Problem statement of one SP region ([MT3] §3.2.1, §3.2.4; [SPN] LayerNorm
 * formula).  Requirements: 1 <= T <= 8; 0 <= j < T; j + nshards <= T;
 * S >= 0, B >= 0, S % T == 0; H > 0 and H % 8 == 0 (bf16) or H % 4 == 0
 * (f32); H <= 16384 (bf16) or 8192 (f32), the longest row the row kernels
 * keep in registers; S*B*H < 2^46; 0 <= p < 1; eps > 0 and finite. */
typedef struct sp_rs_desc_t {
  int32_t T;        /* TP group size = SP group size ([MT3] §3.2.4) */
  int32_t j;        /* first sequence shard processed by this call */
  int64_t S;        /* full sequence length */
  int64_t B;        /* micro-batch */
  int64_t H;        /* hidden size */
  int32_t dtype;    /* sp_dtype_t: activation dtype of every tensor argument */
  int32_t norm;     /* sp_norm_t */
  float p;          /* dropout probability */
  float eps;        /* norm epsilon */
  uint64_t seed;    /* Philox4x32-10 key of the dropout mask */
  int32_t nshards;  /* shards j .. j+nshards-1 in one call; 0 is read as 1 */
  int32_t reserved; /* must be 0 */
  uint32_t* status; /* optional DEVICE word, or NULL; see "Device status" below */
} sp_rs_desc_t;

/* Device status.  Every wait of a kernel on data in flight (a bulk copy
 * landing in shared memory, a ring stage being released) is bounded: after
 * about two seconds the waiting threads give up, mark the results they could
 * not compute (NaN in rstd for the forward's unfinished rows, NaN in every
 * dgamma/dbeta element for the backward), let the copies they started land
 * and return, so the GPU and the CUDA context stay usable.  When desc->status
 * is not NULL, such a kernel also ORs one of the bits below into that 4-byte
 * aligned device word (atomically).  The library never clears the word: the
 * caller zeroes it, runs any number of calls and reads it back whenever it
 * likes (e.g. once per training step).  A clean run leaves it unchanged. */
#define SP_DEVICE_FWD_WAIT_TIMEOUT 0x1u /* a forward kernel gave up waiting */
#define SP_DEVICE_BWD_WAIT_TIMEOUT 0x2u /* a backward kernel gave up waiting */

/* Forward of the SP region for sequence shards j .. j+nshards-1.
 *
 *   Y[r,c]  = sum_{t=0}^{T-1} P_t[row j*R + r, c]      reduce half of the
 *             reduce-scatter, fp32, rank order ([MT3] §3.2.1, §3.3.3)
 *   M[r,c]  = Philox4x32-10(key = seed, counter = (g>>2, 0)) word g&3 >= floor(p*2^32),
 *             g = (j*R + r)*H + c  (global element index; 1-byte mask,
 *             [SPN] MLP activation size)
 *   h[r,c]  = residual[r,c] + Y[r,c]*M[r,c]/(1-p)     dropout then residual
 *             add ([MT3] §3.5; [ATL] §1), stored rounded to dtype
 *   y[r,:]  = RMSNorm: gamma * h * rstd, rstd = 1/sqrt(mean(h^2) + eps)
 *             ([MT4] §4.2.1.1, fp32 inside, one rounding at the end)
 *             LayerNorm: gamma * (h - mean) * rstd + beta,
 *             rstd = 1/sqrt(var + eps), population variance ([SPN] formula)
 *             computed from the stored h.
 *
 * partials : host array of T device pointers, each a full [S,B,H] tensor
 *            (16-byte aligned).  Only rows [j*R, (j+nshards)*R) of each are
 *            read, by their global row index: a caller that holds only those
 *            rows of partial t (a rank that received its shard's block of
 *            every partial, [MT3] §3.2.3) passes the address its row 0 would
 *            have, i.e. the block's address minus j*R*H*element bytes.
 * residual : [nshards*R, H] residual stream of those shards.
 * gamma    : [H]; beta: [H] for LayerNorm (ignored for RMSNorm).
 * h_out, y_out : [nshards*R, H] outputs (residual stream, norm output).
 * mask_out : [nshards*R, H] bytes (0/1), or NULL: then the mask is not
 *            stored and the backward regenerates it from the seed.
 * rstd_out : [nshards*R] fp32.  mean_out: [nshards*R] fp32, LayerNorm only
 *            (ignored for RMSNorm).
 * Alignment: activation pointers and mask 16 bytes; rstd/mean 4 bytes.
 * With no rows to process (S == 0 or B == 0) the call returns SP_OK at once
 * and no pointer is checked or touched. */
sp_status_t sp_rs_dropout_residual_norm_fwd(const sp_rs_desc_t* desc,
                                            const void* const* partials,
                                            const void* residual,
                                            const void* gamma, const void* beta,
                                            void* h_out, void* y_out,
                                            uint8_t* mask_out,
                                            float* rstd_out, float* mean_out,
                                            sp_stream_t stream);

/* The forward above restricted to rows [row_begin, row_begin + row_count)
 * of the call's nshards*R rows: the receiving side of a reduce-scatter split
 * into pipeline chunks, where each chunk's reduction runs as soon as the
 * chunk has arrived while the next chunks are still in flight ([SPN]
 * communication-computation overlap, reduce-scatter overlap by pipeline
 * chunks, 4 by default; [MT3] §3.2.3).  Every argument means what it means
 * in sp_rs_dropout_residual_norm_fwd: residual, h_out, y_out, mask_out,
 * rstd_out and mean_out address the call's row 0 and the partials are
 * addressed by global row, so a caller that holds only a chunk's rows of
 * partial t passes the address that chunk's rows imply for the partial's
 * row 0 (the chunk buffer's address minus (j*R + row_begin)*H*element bytes).
 * Only the rows of the range are read and written, and each of them comes
 * out bit-identical to the full call's (the mask is keyed by the global
 * element index).
 * Errors: as the full call; besides, SP_ERR_INVALID_ARG unless
 * 0 <= row_begin <= row_begin + row_count <= nshards*R, and SP_ERR_ALIGN when
 * the range's first row breaks the 16-byte alignment of the activation or
 * mask pointers (row_begin*H must be a multiple of 16 when a mask is
 * stored).  row_count == 0 returns SP_OK without checking the pointers. */
sp_status_t sp_rs_dropout_residual_norm_fwd_rows(const sp_rs_desc_t* desc,
                                                 int64_t row_begin, int64_t row_count,
                                                 const void* const* partials,
                                                 const void* residual, const void* gamma,
                                                 const void* beta, void* h_out, void* y_out,
                                                 uint8_t* mask_out,
                                                 float* rstd_out, float* mean_out,
                                                 sp_stream_t stream);

/* Bytes of device workspace sp_rs_dropout_residual_norm_bwd needs for this
 * problem on the CURRENT device (it depends on the SM count).  Returns 0 for
 * an invalid descriptor. */
size_t sp_rs_bwd_workspace_bytes(const sp_rs_desc_t* desc);

/* Backward of the SP region for shards j .. j+nshards-1.
 *
 *   g      = gamma * dy
 *   RMS:   xhat = h*rstd,          dh = rstd*(g - xhat*mean(g*xhat))
 *   LN:    xhat = (h-mean)*rstd,   dh = rstd*(g - mean(g) - xhat*mean(g*xhat))
 *   dH     = dh + dh_out                                (dh_out may be NULL)
 *   d_residual = dH                    (the residual add passes dH on)
 *   d_sum  = dH * M / (1-p)            (dropout backward needs only M,
 *                                       [SPN] MLP activation size)
 *   d_sum is the gradient of the reduced sum and so of each partial P_t on
 *   these rows: the all-gather of the backward followed by the add node's
 *   copy ([MT3] §3.3.3.1) needs no T copies on one GPU.
 *   dgamma[c] = sum_r dy[r,c]*xhat[r,c];  dbeta[c] = sum_r dy[r,c]
 *   over the processed rows only: the sum over shards is the all-reduce of
 *   replicated-parameter gradients ([MT3] §3.4.2.1), which a call with
 *   nshards = T performs in place.  Deterministic two-pass reduction.
 *
 * dy, dh_out, h_saved : [nshards*R, H]; gamma: [H]; mask: [nshards*R, H]
 * bytes as written by the forward, or NULL: with p > 0 the keep decisions
 * are then recomputed from desc->seed and the global element index -- the
 * same generator stream, so bit-identical to a stored mask -- trading
 * 2 bytes per element of mask traffic (forward write, backward read) for
 * the generator's arithmetic; rstd, mean: [nshards*R] as written by the forward
 * (mean ignored for RMSNorm).  d_residual, d_sum: [nshards*R, H] outputs;
 * dgamma, dbeta: [H] fp32 outputs (dbeta ignored for RMSNorm).
 * workspace: device scratch of at least sp_rs_bwd_workspace_bytes(desc)
 * bytes, 16-byte aligned; its contents need no initialisation and are
 * meaningless afterwards.  With no rows to process only dgamma (and dbeta)
 * are required; they are set to zero. */
sp_status_t sp_rs_dropout_residual_norm_bwd(const sp_rs_desc_t* desc,
                                            const void* dy, const void* dh_out,
                                            const void* h_saved, const void* gamma,
                                            const uint8_t* mask,
                                            const float* rstd, const float* mean,
                                            void* d_residual, void* d_sum,
                                            float* dgamma, float* dbeta,
                                            void* workspace, size_t workspace_bytes,
                                            sp_stream_t stream);

/* The backward above restricted to rows [row_begin, row_begin + row_count)
 * of the call's nshards*R rows, so that a rank can pass on each chunk of its
 * shard's d_sum (the all-gather that is the backward of the reduce-scatter,
 * [MT3] §3.3.3.1) while the next chunk is still being computed ([SPN]
 * communication-computation overlap).  Every argument means what it means in
 * sp_rs_dropout_residual_norm_bwd: the per-row arguments address the call's
 * row 0, and only the rows of the range are read and written, each of them
 * bit-identical to the full call's.  dgamma/dbeta receive the sums over the
 * range's rows; with accumulate != 0 they are added to what dgamma/dbeta
 * hold (in a fixed order, so the chunks of a shard run in sequence on one
 * stream give a deterministic result that equals the full call's up to the
 * grouping of the sum), else they replace it.  The workspace of the full
 * call suffices for any range.
 * Errors: as the full call; besides, SP_ERR_INVALID_ARG unless
 * 0 <= row_begin <= row_begin + row_count <= nshards*R, and SP_ERR_ALIGN when
 * the range's first row breaks the 16-byte alignment of the activation or
 * mask pointers.  row_count == 0 writes zeros to dgamma/dbeta, or with
 * accumulate != 0 launches nothing. */
sp_status_t sp_rs_dropout_residual_norm_bwd_rows(const sp_rs_desc_t* desc,
                                                 int64_t row_begin, int64_t row_count,
                                                 int32_t accumulate,
                                                 const void* dy, const void* dh_out,
                                                 const void* h_saved, const void* gamma,
                                                 const uint8_t* mask,
                                                 const float* rstd, const float* mean,
                                                 void* d_residual, void* d_sum,
                                                 float* dgamma, float* dbeta,
                                                 void* workspace, size_t workspace_bytes,
                                                 sp_stream_t stream);

/* Size of the fixed device scratch of sp_rs_dropout_residual_norm_bwd_noalloc. */
#define SP_NOALLOC_SCRATCH_BYTES (8u << 20)

/* The backward above without a workspace argument.  The pages have no
 * counterpart to this entry point; it is here for callers that cannot
 * allocate device memory at the point where they run the backward: code
 * inside an allocator callback or an out-of-memory handler (allocating there
 * would re-enter the allocator), frameworks whose caching allocator already
 * holds the device memory and must not see cudaMalloc called behind its
 * back, and latency-critical paths that avoid cudaMalloc / cudaFree because
 * those calls can synchronise the device.
 *
 * Instead of `workspace`, the call uses a fixed array of
 * SP_NOALLOC_SCRATCH_BYTES (8 MiB) in the library's own device memory; every
 * GPU that loads the library reserves it until the process exits.  Arguments,
 * results and errors are those of sp_rs_dropout_residual_norm_bwd, except that
 * a problem whose dgamma/dbeta partial rows need more than
 * SP_NOALLOC_SCRATCH_BYTES (sp_rs_bwd_workspace_bytes(desc) larger than it)
 * is refused with SP_ERR_WORKSPACE before anything is launched.  The call
 * itself allocates nothing.
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it; make that first call before any stream
 * capture begins.  All calls share the one array, which keeps whatever the
 * previous call left in it; nothing in it has to start at zero, because each
 * call writes every partial row it later reads.  Calls whose kernels can
 * overlap on the GPU (different streams, or host threads without ordering)
 * race on the array: order them on one stream. */
sp_status_t sp_rs_dropout_residual_norm_bwd_noalloc(const sp_rs_desc_t* desc,
                                                    const void* dy, const void* dh_out,
                                                    const void* h_saved, const void* gamma,
                                                    const uint8_t* mask,
                                                    const float* rstd, const float* mean,
                                                    void* d_residual, void* d_sum,
                                                    float* dgamma, float* dbeta,
                                                    sp_stream_t stream);

/* sp2hp ([ATL] §5): sequence-split -> hidden-split.  `in` is [N, H]: the T
 * rank shards [N/T, H] stacked in rank order; `out` is [T][N][H/T] where
 * out[r] is what rank r holds after the all-to-all:
 *   out[r][n][c] = in[n][r*H/T + c].
 * Requirements: N % T == 0, (H/T) % 8 == 0 (bf16) or % 4 == 0 (f32),
 * 1 <= T <= 8, both pointers 16-byte aligned.  Bit-exact copy. */
sp_status_t sp2hp(const void* in, void* out, int64_t N, int64_t H, int32_t T,
                  int32_t dtype, sp_stream_t stream);

/* hp2sp ([ATL] §5): the inverse, out[n][r*H/T + c] = in[r][n][c]. */
sp_status_t hp2sp(const void* in, void* out, int64_t N, int64_t H, int32_t T,
                  int32_t dtype, sp_stream_t stream);

/* Static string for a status code. */
const char* sp_status_string(sp_status_t status);

/* Text of the CUDA error behind the most recent SP_ERR_CUDA returned to the
 * calling host thread ("no error" if there was none). */
const char* sp_last_cuda_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int32_t sp_version(void);

/* SHA-256 (hex) of the sources the library was built from, so a binding can
 * refuse a library that does not match its tree. */
const char* sp_build_hash(void);

/* The launch configuration of one TMA-fed kernel (all fields 0 when the
 * register-resident kernel would run instead).  Sizes in bytes. */
typedef struct sp_kernel_plan_t {
  int32_t tma;            /* 1: TMA-fed kernel, 0: register-resident kernel */
  int32_t block;          /* threads launched per CTA (row groups + producer warp) */
  int32_t nthr;           /* block size the kernel's registers are budgeted for */
  int32_t tpr;            /* threads per token row */
  int32_t vpt;            /* 16-byte vectors of the row per thread */
  int32_t row_groups;     /* rows a CTA works on at the same time */
  int32_t rows_per_stage; /* rows per shared-memory ring stage (1 when chunked) */
  int32_t stages;         /* ring stages */
  int32_t chunked;        /* forward only: a stage holds one column chunk of a row */
  int32_t noalloc_fits;   /* backward only: 1 when workspace_bytes fits the fixed scratch of
                             sp_rs_dropout_residual_norm_bwd_noalloc (which refuses the call
                             otherwise), 0 when it does not */
  int64_t stage_bytes;    /* one ring stage, all inputs */
  int64_t smem_bytes;     /* dynamic shared memory per CTA */
  int64_t rows_per_cta;   /* contiguous token rows each CTA owns */
  int64_t ctas;           /* grid size */
  int64_t workspace_bytes; /* backward only: sp_rs_bwd_workspace_bytes on such a device */
} sp_kernel_plan_t;

typedef struct sp_plan_info_t {
  sp_kernel_plan_t fwd;
  sp_kernel_plan_t bwd;
} sp_plan_info_t;

/* What sp_rs_dropout_residual_norm_fwd / _bwd would launch for `desc` on a
 * device with `sms` multiprocessors and `smem_optin` bytes of opt-in shared
 * memory per block (the two values the calls read from the current device),
 * for a backward with or without dh_out and a stored mask.  Host arithmetic
 * only: needs no GPU and launches nothing.  `out` is caller-owned.  Errors:
 * the descriptor's, SP_ERR_INVALID_ARG for a NULL `out` or non-positive
 * limits. */
sp_status_t sp_plan_describe(const sp_rs_desc_t* desc, int32_t sms, int32_t smem_optin,
                             int32_t has_dh, int32_t has_mask, sp_plan_info_t* out);

#ifdef __cplusplus
}
#endif
#endif /* SPFUSE_H */
