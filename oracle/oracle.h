/*
 * oracle.h -- plain, slow, single-threaded fp64 CPU oracle for the
 * sequence-parallel (SP) region hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this library; only the test suite, the smoke check and the
 * bench's CPU-baseline leg do.  It shares no source with the CUDA library.
 *
 * What it computes (sources are the four pages on Megatron-style sequence
 * parallelism this project follows):
 *  - reduce half of reduce-scatter: Y^(j) = sum_t P_t^(j)
 *      MiniMind-tron ch.3 "Sequence Parallelism: layout and gradients",
 *      §3.2.1 (block form of all-reduce = reduce-scatter + all-gather)
 *  - dropout with a stored 0/1 byte mask, Z = Z' (.) M
 *      "Sequence Parallel" notes (cloudchewie), section "MLP activation size"
 *  - residual add, then RMSNorm (fp32-internal in the product, fp64 here) or
 *    LayerNorm gamma*(x-mu)/sqrt(var+eps)+beta
 *      "Sequence Parallel" notes, LayerNorm formula;
 *      MiniMind-tron ch.4, §4.2.1.1 (RMSNorm line)
 *  - the backward of that chain, with the gradient of every partial equal to
 *    the gathered gradient (add node copies its gradient)
 *      MiniMind-tron ch.3, §3.3.3.1
 *  - sp2hp / hp2sp layout transforms (split + all-to-all + cat)
 *      LLM Infra Atlas "03 · Sequence Parallelism", §5
 *  - simulated collectives over T rank buffers, including the ring
 *    reduce-scatter schedule of MiniMind-tron ch.3, §3.2.3
 *
 * Storage types: ORC_F32 / ORC_BF16 are the activation dtypes of the product;
 * ORC_F64 stores unrounded doubles and exists so that pins (finite
 * differences, exact sums) can run the same arithmetic without rounding.
 * Every store rounds exactly once, f64 -> dtype, round-to-nearest-even.
 */
#ifndef SP_ORACLE_H
#define SP_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };
enum { ORC_RMS = 0, ORC_LN = 1 };

typedef struct {
  int32_t T;        /* tensor/sequence parallel group size */
  int32_t j;        /* first sequence shard processed */
  int32_t nshards;  /* consecutive shards processed (>= 1) */
  int32_t dtype;    /* ORC_F32, ORC_BF16 or ORC_F64 */
  int32_t norm;     /* ORC_RMS or ORC_LN */
  int32_t pad;
  int64_t S, B, H;  /* full sequence length, micro-batch, hidden size */
  double p;         /* dropout probability, 0 <= p < 1 */
  double eps;       /* norm epsilon */
  uint64_t seed;    /* Philox key */
} orc_problem;

/* ---- scalar conversions ------------------------------------------------ */
double orc_f64_from_bf16(uint16_t b);
uint16_t orc_bf16_from_f64(double x);          /* direct RNE, no f32 step */
double orc_load(int32_t dtype, const void* base, int64_t idx);
void orc_store(int32_t dtype, void* base, int64_t idx, double v);
int32_t orc_elem_bytes(int32_t dtype);

/* ---- counter-based RNG (Philox4x32-10, Salmon et al., SC'11) ----------- */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
/* word (g & 3) of Philox4x32-10 with key = (lo32 seed, hi32 seed) and
 * counter = (lo32(g>>2), hi32(g>>2), 0, 0) */
uint32_t orc_mask_word(uint64_t seed, uint64_t g);
uint32_t orc_keep_threshold(double p);          /* floor(p * 2^32) */
uint8_t orc_keep(uint64_t seed, uint32_t thr, uint64_t g);

/* ---- forward ------------------------------------------------------------ */
/* One token row.  grow = global row index in the [S*B] rows of the full
 * tensor; prow[t] points at that row (H elements) of partial t; res_row at
 * the residual row.  Outputs: the rounded h and y rows, the mask row, the
 * row statistics and the unrounded values (h before its single rounding, y
 * before its single rounding, the latter computed from the ROUNDED h).
 * Any output pointer may be NULL. */
void orc_fwd_row(const orc_problem* pr, int64_t grow, const void* const* prow,
                 const void* res_row, const void* gamma, const void* beta,
                 void* h_row, void* y_row, uint8_t* mask_row, double* rstd,
                 double* mean, double* h_exact, double* y_exact);

/* Shards j .. j+nshards-1: rows [j*R, (j+nshards)*R), R = (S/T)*B.
 * partials: T pointers to full [S,B,H] tensors.  residual and all row
 * outputs are [nshards*R, H]; rstd/mean are [nshards*R].  Returns 0 or a
 * negative error code for an invalid problem. */
int orc_fwd(const orc_problem* pr, const void* const* partials,
            const void* residual, const void* gamma, const void* beta,
            void* h_out, void* y_out, uint8_t* mask_out, double* rstd_out,
            double* mean_out, double* h_exact, double* y_exact);

/* ---- backward ----------------------------------------------------------- */
/* One row.  Row statistics are recomputed in f64 from h_row.  dh_row may be
 * NULL (no gradient from the residual stream); mask_row may be NULL only
 * when p == 0.  dgamma_acc / dbeta_acc (H doubles, may be NULL) receive
 * += the row's contribution. */
void orc_bwd_row(const orc_problem* pr, const void* dy_row, const void* dh_row,
                 const void* h_row, const void* gamma, const uint8_t* mask_row,
                 void* dres_row, void* dsum_row, double* dres_exact,
                 double* dsum_exact, double* dgamma_acc, double* dbeta_acc);

/* All rows of shards j .. j+nshards-1; dgamma/dbeta are the sums over
 * those rows (written, not accumulated). */
int orc_bwd(const orc_problem* pr, const void* dy, const void* dh_out,
            const void* h_saved, const void* gamma, const uint8_t* mask,
            void* d_residual, void* d_sum, double* dres_exact,
            double* dsum_exact, double* dgamma, double* dbeta);

/* Row statistics of one stored row, f64: rstd = 1/sqrt(var + eps) (LN) or
 * 1/sqrt(mean(h^2) + eps) (RMS); mean = mu (LN) or 0 (RMS). */
void orc_norm_stats_row(const orc_problem* pr, const void* h_row, double* rstd, double* mean);

/* Array helpers for the bindings: n conversions, each one rounding. */
void orc_bf16_from_f64_array(const double* x, uint16_t* out, int64_t n);
void orc_f64_from_bf16_array(const uint16_t* x, double* out, int64_t n);
/* keep bits for n consecutive global indices g0 .. g0+n-1 */
void orc_mask_range(uint64_t seed, double p, uint64_t g0, int64_t n, uint8_t* out);

/* ---- simulated collectives over T rank buffers (f64) -------------------- */
/* Each rank buffer has n elements, split along dim 0 into T equal blocks. */
int orc_reduce_scatter(int32_t T, int64_t n, const double* const* P, int32_t j, double* out);
int orc_all_gather(int32_t T, int64_t m, const double* const* blocks, double* out);
int orc_all_reduce(int32_t T, int64_t n, const double* const* P, double* out);
/* Ring reduce-scatter on running partials work[t] (modified in place).
 * After T-1 steps rank t's block t holds the full sum.  sent[t] counts the
 * elements rank t sent. */
int orc_ring_reduce_scatter(int32_t T, int64_t n, double* const* work, int64_t* sent);
/* Same schedule on contributor sets: contrib[r*T+b] is the bit set of
 * original ranks summed in rank r's cell for block b, used[r*T+b] is 1 once
 * rank r has sent that cell.  Runs `steps` steps from the initial state. */
int orc_ring_reduce_scatter_symbolic(int32_t T, int32_t steps, uint64_t* contrib, uint8_t* used);

/* ---- layout transforms (bytes; elem_bytes = 2 or 4 or 8) ----------------- */
/* sp2hp: in [N,H] (T rank shards stacked in rank order) -> out [T][N][H/T]
 * hp2sp: the inverse. */
int orc_sp2hp(const void* in, void* out, int64_t N, int64_t H, int32_t T, int32_t elem_bytes);
int orc_hp2sp(const void* in, void* out, int64_t N, int64_t H, int32_t T, int32_t elem_bytes);
/* The same two maps built the way the pages describe them: split along one
 * dim, exchange piece s of rank r to rank s, concatenate along the other. */
int orc_sp2hp_all_to_all(const void* in, void* out, int64_t N, int64_t H, int32_t T, int32_t elem_bytes);
int orc_hp2sp_all_to_all(const void* in, void* out, int64_t N, int64_t H, int32_t T, int32_t elem_bytes);

#ifdef __cplusplus
}
#endif
#endif
