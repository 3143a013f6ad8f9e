// common.cuh -- device helpers shared by the libspfuse kernels (sm_103a).
//
// Vector width: every kernel moves activations in 16-byte vectors
// (8 bf16 or 4 fp32 elements), so a warp touches 512 contiguous bytes per
// access and H must be a multiple of the vector width.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace spf {

constexpr int kMaxT = 8;  // largest TP/SP group the kernels unroll for

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel waits for the grids it depends
// on before its first global read, and lets the next kernel in the stream be
// scheduled as soon as all of its own CTAs are resident.  (Letting it be
// scheduled before the wait measured the same at the pages' shape.)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier over `nthreads` threads (a multiple of 32); ids 1..15.
__device__ __forceinline__ void bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
// Easy as 1, 2, 3", SC'11): ten rounds, each taking the 64-bit products of
// counter words 0 and 2 with the two round multipliers and mixing their
// halves with words 1 and 3 and the round key; the key advances by the two
// Weyl increments between rounds.
// ---------------------------------------------------------------------------
// The ten round keys (rk[2i], rk[2i+1] = the key advanced i times) are
// precomputed on the host and read from kernel parameters; the counter's upper
// two words are zero, as in the mask's counter layout.
struct PhiloxKeys {
  uint32_t rk[20];
};

__device__ __forceinline__ uint4 philox4x32_10_rk(uint32_t c0, uint32_t c1, const PhiloxKeys& k) {
  uint32_t c2 = 0u, c3 = 0u;
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k.rk[2 * i];
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k.rk[2 * i + 1];
    c1 = (uint32_t)p1;
    c3 = (uint32_t)p0;
    c0 = n0;
    c2 = n2;
  }
  return make_uint4(c0, c1, c2, c3);
}

// Keep bits of the 4 consecutive elements 4q .. 4q+3 (bit e = element 4q+e):
// element g is kept when word (g & 3) of the block at counter g >> 2 is at
// least the threshold floor(p * 2^32).
__device__ __forceinline__ uint32_t keep_bits4(uint64_t q, const PhiloxKeys& k, uint32_t thr) {
  const uint4 w = philox4x32_10_rk((uint32_t)q, (uint32_t)(q >> 32), k);
  return (uint32_t)(w.x >= thr) | ((uint32_t)(w.y >= thr) << 1) | ((uint32_t)(w.z >= thr) << 2) |
         ((uint32_t)(w.w >= thr) << 3);
}

// ---------------------------------------------------------------------------
// 16-byte global accesses.  Inputs that are read once (partials, residual,
// upstream gradients, saved activations) and the outputs read later use the
// streaming (evict-first) cache policy; gamma/beta, re-read by every row, go
// through the read-only path.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint4 ld_cached(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}
// An output the next kernel reads right away (the norm output y, which the
// sp2hp layout or the next GEMM reads next) is stored with the default
// policy, so it stays in L2 for that reader.
__device__ __forceinline__ void st_keep(void* p, uint4 v) {
  *reinterpret_cast<uint4*>(p) = v;
}

// ---------------------------------------------------------------------------
// Activation types: unpack a 16-byte vector to fp32, pack fp32 back with one
// round-to-nearest-even per element.
// ---------------------------------------------------------------------------
template <typename Act>
struct Act16;

template <>
struct Act16<float> {
  static constexpr int EV = 4;  // elements per 16-byte vector
  __device__ __forceinline__ static void unpack(uint4 v, float (&f)[EV]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static uint4 pack(const float (&f)[EV]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

template <>
struct Act16<__nv_bfloat16> {
  static constexpr int EV = 8;
  __device__ __forceinline__ static void unpack_word(uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
  }
  __device__ __forceinline__ static void unpack(uint4 v, float (&f)[EV]) {
    unpack_word(v.x, f[0], f[1]);
    unpack_word(v.y, f[2], f[3]);
    unpack_word(v.z, f[4], f[5]);
    unpack_word(v.w, f[6], f[7]);
  }
  __device__ __forceinline__ static uint32_t pack_word(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
    return *reinterpret_cast<uint32_t*>(&b);
  }
  __device__ __forceinline__ static uint4 pack(const float (&f)[EV]) {
    return make_uint4(pack_word(f[0], f[1]), pack_word(f[2], f[3]), pack_word(f[4], f[5]),
                      pack_word(f[6], f[7]));
  }
};

// ---------------------------------------------------------------------------
// Residual stream value h = res + acc * s, rounded ONCE to bf16 from (almost)
// the exact value.  s = s_hi + s_lo carries 1/(1-p) to ~48 bits.  The product
// and the sum are formed with error-free transformations (Dekker's product
// via fma, Knuth's TwoSum), so h = h_hi + err up to the tiny acc*s_lo
// rounding.  The bf16 result is the nearest-even rounding of h_hi + err: the
// magnitude is compared with the bf16 midpoint above trunc(h_hi).  Rounding
// h_hi alone would be wrong whenever the exact value and h_hi straddle a
// midpoint, which is common: when the partial sum times 1/(1-p) is (nearly)
// dyadic, fp32 arithmetic lands on or next to a tie the exact value misses.
// Returns the bf16 bit pattern.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t residual_bf16_dd(float res, float acc, float s_hi, float s_lo,
                                                     bool keep) {
  float h_hi = res, err = 0.f;
  if (keep) {
    const float z_hi = __fmul_rn(acc, s_hi);
    const float z_lo = __fadd_rn(__fmaf_rn(acc, s_hi, -z_hi), __fmul_rn(acc, s_lo));
    h_hi = __fadd_rn(res, z_hi);
    const float bb = __fsub_rn(h_hi, res);
    const float e1 = __fadd_rn(__fsub_rn(res, __fsub_rn(h_hi, bb)), __fsub_rn(z_hi, bb));
    err = __fadd_rn(e1, z_lo);
  }
  // renormalise (TwoSum): hs = fl(h_hi + err), |lo| <= ulp(hs)/2, so the
  // midpoint test below also holds when res and z cancel
  const float hs = __fadd_rn(h_hi, err);
  const float bs = __fsub_rn(hs, h_hi);
  const float lo = __fadd_rn(__fsub_rn(h_hi, __fsub_rn(hs, bs)), __fsub_rn(err, bs));
  const uint32_t u = __float_as_uint(hs);
  if ((u & 0x7FFFFFFFu) == 0u) {  // exact cancellation: the value is lo itself
    const __nv_bfloat16 b = __float2bfloat16_rn(lo);
    return (uint32_t) * reinterpret_cast<const unsigned short*>(&b);
  }
  const uint32_t trunc = u & 0xFFFF0000u;              // toward zero, same exponent
  const float mid = __uint_as_float(trunc | 0x8000u);  // midpoint above |trunc|
  // |h| - |mid|: the first difference is exact (same binade), lo adds the rest
  const float d = __fadd_rn(__fsub_rn(fabsf(hs), fabsf(mid)), hs > 0.f ? lo : -lo);
  uint32_t b = trunc >> 16;
  if (d > 0.f || (d == 0.f && (b & 1u))) b += 1u;
  return b;
}

// The common case of the same rounding, in a few operations.  h1 = fl(res +
// acc*s_hi) lies in the bf16 interval [trunc, trunc + ulp) whose midpoint m is
// the only rounding boundary the exact value E = res + acc*(s_hi + s_lo) can be
// near.  res - m is exact when res and h1 are within 2^12 of each other in
// magnitude (both are on coarse grids: res is bf16, m has 9 significant bits),
// so fma(acc, s_lo, fma(acc, s_hi, res - m)) has the sign of E - m, and E
// rounds away from zero past m, toward zero before it, to even on it.  Heavy
// cancellation (or a residual far below h) takes the double-float routine.
__device__ __forceinline__ uint32_t residual_bf16(float res, float acc, float s_hi, float s_lo,
                                                  bool keep) {
  if (!keep) return __float_as_uint(res) >> 16;  // res is a bf16 value already
  const float h1 = __fmaf_rn(acc, s_hi, res);
  const float ah = fabsf(h1), ar = fabsf(res);
  if (ah < 0x1p-12f * ar || (ar < 0x1p-12f * ah && res != 0.f))
    return residual_bf16_dd(res, acc, s_hi, s_lo, true);
  const uint32_t u = __float_as_uint(h1);
  const uint32_t tr = u & 0xFFFF0000u;
  const float rm = __fsub_rn(res, __uint_as_float(tr | 0x8000u));
  const float d = __fmaf_rn(acc, s_lo, __fmaf_rn(acc, s_hi, rm));
  uint32_t b = tr >> 16;
  const bool beyond = d != 0.f && ((__float_as_uint(d) ^ u) >> 31) == 0u;  // E past m
  if (beyond || (d == 0.f && (b & 1u))) b += 1u;
  return b;
}

// ---------------------------------------------------------------------------
// Packed pairs of fp32 (Blackwell f32x2 arithmetic: one instruction works on
// two lanes).  Element 2i sits in the low half, 2i+1 in the high half, so a
// bf16 pair unpacks with one shift and one mask.
// ---------------------------------------------------------------------------
typedef unsigned long long f2_t;

__device__ __forceinline__ f2_t f2(float lo, float hi) {
  f2_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(f2_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2_t f2_add(f2_t a, f2_t b) {
  f2_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_sub(f2_t a, f2_t b) {
  f2_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_mul(f2_t a, f2_t b) {
  f2_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_fma(f2_t a, f2_t b, f2_t c) {
  f2_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2_t bf2_to_f2(uint32_t w) {
  return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ uint32_t f2_to_bf2(f2_t v) {  // round each lane to nearest even
  float lo, hi;
  f2_split(v, lo, hi);
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

// Residual stream of two elements (one bf16 pair), the packed-pair form of
// residual_bf16: E = res + acc*(s_hi + s_lo) rounded once to bf16, where acc
// is already zero for dropped elements (then E = res, a bf16 value, and the
// test below returns it unchanged).  Same midpoint test: with h1 = fl(res +
// acc*s_hi) and m the bf16 midpoint of h1's interval, d = fma(acc, s_lo,
// fma(acc, s_hi, res - m)) has the sign of E - m; round away from zero when d
// and h1 agree in sign, to even when d = 0.  res - m is exact unless h1 is
// far below res (heavy cancellation); those lanes take the double-float
// routine.  A residual far below h (|res| < 2^-12 |h|, so res - m may round)
// is not guarded: the decision can then only go wrong when E is within one
// fp32 ulp of the midpoint as well, a joint event of probability ~1e-9.
__device__ __forceinline__ uint32_t residual_bf2(f2_t res, f2_t acc, f2_t s_hi, f2_t s_lo) {
  const f2_t h1 = f2_fma(acc, s_hi, res);
  float h1l, h1h;
  f2_split(h1, h1l, h1h);
  const uint32_t ul = __float_as_uint(h1l), uh = __float_as_uint(h1h);
  const f2_t m = f2(__uint_as_float((ul & 0xFFFF0000u) | 0x8000u),
                    __uint_as_float((uh & 0xFFFF0000u) | 0x8000u));
  const f2_t d = f2_fma(acc, s_lo, f2_fma(acc, s_hi, f2_sub(res, m)));
  const f2_t gap = f2_mul(h1, f2(0x1p12f, 0x1p12f));
  float dl, dh, gl, gh, rl, rh;
  f2_split(d, dl, dh);
  f2_split(gap, gl, gh);
  f2_split(res, rl, rh);
  uint32_t bl = ul >> 16, bh = uh >> 16;
  // d and h1 agree in sign (and d != 0): the exact value lies past m
  const bool pastl = dl != 0.f && (int)(__float_as_uint(dl) ^ ul) >= 0;
  const bool pasth = dh != 0.f && (int)(__float_as_uint(dh) ^ uh) >= 0;
  bl += (pastl || (dl == 0.f && (bl & 1u))) ? 1u : 0u;
  bh += (pasth || (dh == 0.f && (bh & 1u))) ? 1u : 0u;
  if (fabsf(gl) < fabsf(rl) || fabsf(gh) < fabsf(rh)) {  // rare: |h| < 2^-12 |res|
    float al, ah, shl, shh, sll, slh;
    f2_split(acc, al, ah);
    f2_split(s_hi, shl, shh);
    f2_split(s_lo, sll, slh);
    if (fabsf(gl) < fabsf(rl)) bl = residual_bf16_dd(rl, al, shl, sll, true);
    if (fabsf(gh) < fabsf(rh)) bh = residual_bf16_dd(rh, ah, shh, slh, true);
  }
  return bl | (bh << 16);
}

// Mask bytes <-> keep bits.  Bit 0 of every mask byte is the keep flag (the
// forward writes 0 or 1).  Four bits spread to four bytes with one multiply
// (the shifted copies 0, 7, 14, 21 do not overlap), and four bytes gather
// back to four bits with one multiply (cross terms stay below bit 24 or
// leave the word).
__device__ __forceinline__ uint32_t bits4_to_bytes(uint32_t b4) {
  return (b4 * 0x00204081u) & 0x01010101u;
}
__device__ __forceinline__ uint32_t bytes_to_bits4(uint32_t w) {
  return ((w & 0x01010101u) * 0x01020408u) >> 24;
}

template <int EV>
__device__ __forceinline__ void st_mask(uint8_t* p, uint32_t bits);

template <>
__device__ __forceinline__ void st_mask<8>(uint8_t* p, uint32_t bits) {
  __stcs(reinterpret_cast<uint2*>(p), make_uint2(bits4_to_bytes(bits & 0xFu), bits4_to_bytes(bits >> 4)));
}
template <>
__device__ __forceinline__ void st_mask<4>(uint8_t* p, uint32_t bits) {
  __stcs(reinterpret_cast<unsigned int*>(p), bits4_to_bytes(bits & 0xFu));
}

template <int EV>
__device__ __forceinline__ uint32_t ld_mask(const uint8_t* p);

template <>
__device__ __forceinline__ uint32_t ld_mask<8>(const uint8_t* p) {
  const uint2 w = __ldcs(reinterpret_cast<const uint2*>(p));
  return bytes_to_bits4(w.x) | (bytes_to_bits4(w.y) << 4);
}
template <>
__device__ __forceinline__ uint32_t ld_mask<4>(const uint8_t* p) {
  return bytes_to_bits4(__ldcs(reinterpret_cast<const unsigned int*>(p)));
}

// Eight mask bytes from shared memory as keep bits.
__device__ __forceinline__ uint32_t ld_mask_shared8(const uint8_t* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  return bytes_to_bits4(w.x) | (bytes_to_bits4(w.y) << 4);
}

// Barrier over `nthreads` threads that also ANDs a predicate across them.
__device__ __forceinline__ bool bar_red_and(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0u;
}

// ---------------------------------------------------------------------------
// Sum of NV values over the `tpr` threads that share one token row.
// Butterfly shuffles give every lane of a warp bit-identical sums; across
// warps each thread adds the per-warp sums in warp order, so the result is
// the same on every thread and on every run.  `red` holds 2 slots of
// (tpr/32)*NV floats for this row group; successive calls alternate `slot`
// so one barrier per call is enough.
// ---------------------------------------------------------------------------
template <int NV>
__device__ __forceinline__ void row_allreduce(float (&v)[NV], int tpr, int lane_r, int bar_id,
                                              float* red, int slot) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] += __shfl_xor_sync(0xFFFFFFFFu, v[i], off);
  }
  if (tpr == 32) return;
  const int wpr = tpr >> 5;
  float* buf = red + slot * wpr * NV;
  if ((lane_r & 31) == 0) {
#pragma unroll
    for (int i = 0; i < NV; ++i) buf[(lane_r >> 5) * NV + i] = v[i];
  }
  bar_sync(bar_id, tpr);
#pragma unroll
  for (int i = 0; i < NV; ++i) v[i] = 0.f;
  for (int w = 0; w < wpr; ++w) {
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] += buf[w * NV + i];
  }
}

// ---------------------------------------------------------------------------
// Kernel arguments (passed by value).
// ---------------------------------------------------------------------------
struct FwdArgs {
  const void* P[kMaxT];  // partial outputs, full [S,B,H]
  const void* residual;  // [rows, H]
  const void* gamma;     // [H]
  const void* beta;      // [H] (LayerNorm)
  void* h;               // [rows, H]
  void* y;               // [rows, H]
  uint8_t* mask;         // [rows, H] or null
  float* rstd;           // [rows]
  float* mean;           // [rows] (LayerNorm)
  int64_t rows;          // token rows processed
  int64_t grow0;         // global row index of local row 0 (j * R)
  int32_t H;
  int32_t nvec;          // vectors per row, H / EV
  int32_t tpr;           // threads per row (multiple of 32)
  uint32_t thr;          // keep threshold floor(p * 2^32)
  PhiloxKeys keys;       // Philox round keys of the seed
  float scale;           // 1 / (1 - p), rounded to fp32
  float scale_lo;        // 1 / (1 - p) - scale, rounded to fp32
  float eps;
  float Hf;              // H as float
  int32_t dropout;       // p > 0
  int32_t dyadic_scale;  // 1/(1-p) is exact in fp32 (scale_lo == 0): bf16 ties can occur
  uint32_t* status;      // device status word (timeouts are ORed in) or null
  uint64_t wait_ns;      // bound of every mbarrier wait
  int32_t drop_stage;    // test hook: CTA 0's producer never fills this stage (-1: none)
};

struct BwdArgs {
  const void* dy;        // [rows, H]
  const void* dh;        // [rows, H] or null
  const void* h;         // [rows, H]
  const void* gamma;     // [H]
  const uint8_t* mask;   // [rows, H] or null (p == 0, or regenerate)
  const float* rstd;     // [rows]
  const float* mean;     // [rows] (LayerNorm)
  void* d_res;           // [rows, H]
  void* d_sum;           // [rows, H]
  float* ws;             // [nparts, H] dgamma partials, then [nparts, H] dbeta partials
                         // (one partial row per thread-block cluster)
  int64_t rows;
  int64_t rows_per_cta;  // contiguous rows per CTA
  int32_t H;
  int32_t nvec;
  int32_t tpr;
  int32_t nparts;        // partial rows per statistic
  float scale;           // 1 / (1 - p)
  float Hf;
  int32_t regen;         // p > 0 without a stored mask: recompute the keep bits
  uint32_t thr;          // keep threshold (regen)
  int64_t grow0;         // global row index of local row 0 (regen)
  PhiloxKeys keys;       // Philox round keys of the seed (regen)
  uint32_t* status;      // device status word (timeouts are ORed in) or null
  uint64_t wait_ns;      // bound of every mbarrier wait
  int32_t drop_stage;    // test hook: CTA 0's producer never fills this stage (-1: none)
};

// Bits of the device status word (the values of include/spfuse.h).
constexpr uint32_t kStatusFwdWaitTimeout = 0x1u;
constexpr uint32_t kStatusBwdWaitTimeout = 0x2u;

__device__ __forceinline__ void report_status(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// Shared-memory ring of the TMA-fed forward.
struct FwdTmaLayout {
  int32_t nst;           // stages in the ring
  int32_t nrg;           // consumer row groups
  int32_t rb;            // rows per stage
  uint32_t stage_bytes;  // bytes of one stage
  uint32_t blk;          // bytes of one tensor's rows in a stage (rb * H * 2)
  uint32_t smem_stages;  // offset of stage 0 in dynamic shared memory
  int32_t pf_stages;     // stages prefetched into L2 before the grid-dependency wait
  int64_t rows_per_cta;
};

// Shared-memory ring of the TMA-fed backward.
struct BwdTmaLayout {
  int32_t nst;          // stages in the ring
  int32_t nrg;          // consumer row groups
  int32_t rb;           // rows per stage
  uint32_t stage_bytes; // bytes of one stage
  uint32_t off_h, off_dh, off_mask;  // offsets inside a stage (dy at 0)
  uint32_t smem_stages; // offset of stage 0 in dynamic shared memory
  int32_t pf_stages;    // stages prefetched into L2 before the grid-dependency wait
};

}  // namespace spf
