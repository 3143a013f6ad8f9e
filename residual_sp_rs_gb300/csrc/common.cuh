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
// scheduled as soon as all of its own CTAs are resident.
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
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    if (i > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// Keep bits of the 4 consecutive elements 4q .. 4q+3 (bit e = element 4q+e):
// element g is kept when word (g & 3) of the block at counter g >> 2 is at
// least the threshold floor(p * 2^32).
__device__ __forceinline__ uint32_t keep_bits4(uint64_t q, uint32_t k0, uint32_t k1, uint32_t thr) {
  const uint4 w = philox4x32_10(make_uint4((uint32_t)q, (uint32_t)(q >> 32), 0u, 0u), k0, k1);
  return (uint32_t)(w.x >= thr) | ((uint32_t)(w.y >= thr) << 1) | ((uint32_t)(w.z >= thr) << 2) |
         ((uint32_t)(w.w >= thr) << 3);
}

// ---------------------------------------------------------------------------
// 16-byte global accesses.  Inputs that are read once (partials, residual,
// upstream gradients, saved activations) and all outputs use the streaming
// (evict-first) cache policy; gamma/beta, re-read by every row, go through
// the read-only path.
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
__device__ __forceinline__ uint32_t residual_bf16(float res, float acc, float s_hi, float s_lo,
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

// Store EV mask bytes (bit e of `bits` -> byte e).
template <int EV>
__device__ __forceinline__ void st_mask(uint8_t* p, uint32_t bits);

template <>
__device__ __forceinline__ void st_mask<8>(uint8_t* p, uint32_t bits) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    lo |= ((bits >> e) & 1u) << (8 * e);
    hi |= ((bits >> (e + 4)) & 1u) << (8 * e);
  }
  __stcs(reinterpret_cast<uint2*>(p), make_uint2(lo, hi));
}
template <>
__device__ __forceinline__ void st_mask<4>(uint8_t* p, uint32_t bits) {
  uint32_t w = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) w |= ((bits >> e) & 1u) << (8 * e);
  __stcs(reinterpret_cast<unsigned int*>(p), w);
}

// Load EV mask bytes as bits (byte e nonzero -> bit e).
template <int EV>
__device__ __forceinline__ uint32_t ld_mask(const uint8_t* p);

template <>
__device__ __forceinline__ uint32_t ld_mask<8>(const uint8_t* p) {
  const uint2 w = __ldcs(reinterpret_cast<const uint2*>(p));
  uint32_t bits = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    bits |= (((w.x >> (8 * e)) & 0xFFu) != 0u ? 1u : 0u) << e;
    bits |= (((w.y >> (8 * e)) & 0xFFu) != 0u ? 1u : 0u) << (e + 4);
  }
  return bits;
}
template <>
__device__ __forceinline__ uint32_t ld_mask<4>(const uint8_t* p) {
  const unsigned int w = __ldcs(reinterpret_cast<const unsigned int*>(p));
  uint32_t bits = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) bits |= (((w >> (8 * e)) & 0xFFu) != 0u ? 1u : 0u) << e;
  return bits;
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
  uint32_t key0, key1;   // Philox key (seed)
  float scale;           // 1 / (1 - p), rounded to fp32
  float scale_lo;        // 1 / (1 - p) - scale, rounded to fp32
  float eps;
  float Hf;              // H as float
  int32_t dropout;       // p > 0
};

struct BwdArgs {
  const void* dy;        // [rows, H]
  const void* dh;        // [rows, H] or null
  const void* h;         // [rows, H]
  const void* gamma;     // [H]
  const uint8_t* mask;   // [rows, H] or null (p == 0)
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
  int32_t nparts;        // clusters launched (rows of ws per statistic)
  float scale;           // 1 / (1 - p)
  float Hf;
};

}  // namespace spf
