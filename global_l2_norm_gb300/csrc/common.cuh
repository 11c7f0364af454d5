// common.cuh -- building blocks of the clipping kernels: launch constants,
// the grid-barrier words, float-float arithmetic, the element formats and
// the memory-access policies.  Included by gclip.cu only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "internal.hpp"

namespace gclip {


constexpr int kThreads = 256;             // threads per block, every kernel
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 8;                // 16-byte vectors in flight per thread (scaling)
constexpr int kNormUnroll = 8;            // the same in the norm pass
constexpr long long kDefaultTimeoutNs = 1000000000LL;  // grid barrier: 1 s

struct SyncWords {
  unsigned int arrive;  // blocks done with the norm pass in this call
  unsigned int gen;     // bumped once per call when the record is published
  unsigned int work;    // scaling-pass chunks claimed in this call
  unsigned int pad;
};

// ---------------------------------------------------------------------------
// float-float arithmetic: a value hi + lo with |lo| <= ulp(hi) / 2.  The
// explicit _rn intrinsics keep the compiler from contracting or reordering.

struct FF {
  float hi, lo;
};

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  // Knuth's TwoSum: s + e == a + b exactly, for any order of magnitude.
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ FF ff_renorm(float s, float e) {
  FF r;
  r.hi = __fadd_rn(s, e);
  r.lo = __fsub_rn(e, __fsub_rn(r.hi, s));
  return r;
}

__device__ __forceinline__ FF ff_add_f(FF a, float b) {
  float s, e;
  two_sum(a.hi, b, s, e);
  return ff_renorm(s, __fadd_rn(e, a.lo));
}

__device__ __forceinline__ FF ff_add(FF a, FF b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  return ff_renorm(s, __fadd_rn(e, __fadd_rn(a.lo, b.lo)));
}

// ---------------------------------------------------------------------------
// The sum of squares in two bins.  A square is taken in fp32, so an unscaled
// element y = x * inv_scale with |y| < 2^-63 has a subnormal or zero square.
// A vector (or scalar element) whose fp32 sum of squares is at least kTinySq
// goes to `big`; the others go to `tiny` as the squares of x * inv_scale *
// 2^K, with K chosen per call so that inv_scale * 2^K is a finite fp32 number
// (K = 96 unless inv_scale > 2^30).  Both bins are float-float sums; the
// total is big + tiny * 2^-2K, formed in double by the final reduction.  A
// vector in `tiny` has every |y| < 2^-50, so its scaled squares are below
// 2^92 (no overflow over 2^35 vectors), and every |y| >= 2^(-63-K) (2^-159)
// has a normal scaled square: neither bin underflows where it matters.

constexpr float kTinySq = 0x1p-100f;
constexpr int kTinyExpMax = 96;

struct SumSq {
  FF big, tiny;
};

__device__ __forceinline__ SumSq sumsq_add(SumSq a, SumSq b) {
  return SumSq{ff_add(a.big, b.big), ff_add(a.tiny, b.tiny)};
}

// ---------------------------------------------------------------------------
// Element formats.  A 16-byte vector holds 4 fp32 or 8 fp16/bf16 elements,
// element 0 in the lowest bytes.

template <int DT>
struct Fmt;

template <>
struct Fmt<GCLIP_F32> {
  static constexpr int kPerVec = 4;
  static constexpr int kBytes = 4;
  __device__ static __forceinline__ float load1(uint64_t a) {
    return __ldcg(reinterpret_cast<const float*>(a));
  }
  __device__ static __forceinline__ void store1(uint64_t a, float v) {
    *reinterpret_cast<float*>(a) = v;
  }
  // Sum of the four squares of x * k, one rounding per element (the first
  // product, then fused multiply-adds in element order).
  __device__ static __forceinline__ float sumsq(uint4 v, float k) {
    const float y0 = __fmul_rn(__uint_as_float(v.x), k);
    const float y1 = __fmul_rn(__uint_as_float(v.y), k);
    const float y2 = __fmul_rn(__uint_as_float(v.z), k);
    const float y3 = __fmul_rn(__uint_as_float(v.w), k);
    float r = __fmul_rn(y0, y0);
    r = __fmaf_rn(y1, y1, r);
    r = __fmaf_rn(y2, y2, r);
    r = __fmaf_rn(y3, y3, r);
    return r;
  }
  __device__ static __forceinline__ uint4 scale(uint4 v, float chi, float clo) {
    uint4 o;
    o.x = __float_as_uint(scale1(__uint_as_float(v.x), chi, clo));
    o.y = __float_as_uint(scale1(__uint_as_float(v.y), chi, clo));
    o.z = __float_as_uint(scale1(__uint_as_float(v.z), chi, clo));
    o.w = __float_as_uint(scale1(__uint_as_float(v.w), chi, clo));
    return o;
  }
  // x * (chi + clo) rounded once: x * chi is exact inside the fma.
  __device__ static __forceinline__ float scale1(float x, float chi, float clo) {
    return __fmaf_rn(x, chi, __fmul_rn(x, clo));
  }
  // Element-wise x + a of two stored vectors, each sum rounded once.
  __device__ static __forceinline__ uint4 add(uint4 x, uint4 a) {
    return make_uint4(__float_as_uint(__fadd_rn(__uint_as_float(x.x), __uint_as_float(a.x))),
                      __float_as_uint(__fadd_rn(__uint_as_float(x.y), __uint_as_float(a.y))),
                      __float_as_uint(__fadd_rn(__uint_as_float(x.z), __uint_as_float(a.z))),
                      __float_as_uint(__fadd_rn(__uint_as_float(x.w), __uint_as_float(a.w))));
  }
  // A float rounded to the storage format (here: itself).
  __device__ static __forceinline__ float round1(float v) { return v; }
};

template <>
struct Fmt<GCLIP_F16> {
  static constexpr int kPerVec = 8;
  static constexpr int kBytes = 2;
  __device__ static __forceinline__ float2 widen(uint32_t w) {
    __half2 h;
    memcpy(&h, &w, 4);
    return __half22float2(h);
  }
  __device__ static __forceinline__ uint32_t narrow(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    uint32_t w;
    memcpy(&w, &h, 4);
    return w;
  }
  __device__ static __forceinline__ float load1(uint64_t a) {
    const unsigned short u = __ldcg(reinterpret_cast<const unsigned short*>(a));
    return __half2float(__ushort_as_half(u));
  }
  __device__ static __forceinline__ void store1(uint64_t a, float v) {
    *reinterpret_cast<unsigned short*>(a) = __half_as_ushort(__float2half_rn(v));
  }
  // Sum of the eight squares of x * k, as for fp32.
  __device__ static __forceinline__ float sumsq(uint4 v, float k) {
    const float2 a = widen(v.x), b = widen(v.y), c = widen(v.z), d = widen(v.w);
    const float y[8] = {__fmul_rn(a.x, k), __fmul_rn(a.y, k), __fmul_rn(b.x, k),
                        __fmul_rn(b.y, k), __fmul_rn(c.x, k), __fmul_rn(c.y, k),
                        __fmul_rn(d.x, k), __fmul_rn(d.y, k)};
    float r = __fmul_rn(y[0], y[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) r = __fmaf_rn(y[i], y[i], r);
    return r;
  }
  __device__ static __forceinline__ uint32_t scale_word(uint32_t w, float chi, float clo) {
    const float2 f = widen(w);
    return narrow(Fmt<GCLIP_F32>::scale1(f.x, chi, clo),
                  Fmt<GCLIP_F32>::scale1(f.y, chi, clo));
  }
  __device__ static __forceinline__ uint4 scale(uint4 v, float chi, float clo) {
    return make_uint4(scale_word(v.x, chi, clo), scale_word(v.y, chi, clo),
                      scale_word(v.z, chi, clo), scale_word(v.w, chi, clo));
  }
  // Element-wise x + a, each sum rounded once to the format: the float sum
  // of two values of a format with p <= 11 significand bits, rounded again
  // to the format, is the correctly rounded sum (24 >= 2p + 2).
  __device__ static __forceinline__ uint32_t add_word(uint32_t x, uint32_t a) {
    const float2 f = widen(x), g = widen(a);
    return narrow(__fadd_rn(f.x, g.x), __fadd_rn(f.y, g.y));
  }
  __device__ static __forceinline__ uint4 add(uint4 x, uint4 a) {
    return make_uint4(add_word(x.x, a.x), add_word(x.y, a.y), add_word(x.z, a.z),
                      add_word(x.w, a.w));
  }
  __device__ static __forceinline__ float round1(float v) {
    return __half2float(__float2half_rn(v));
  }
};

template <>
struct Fmt<GCLIP_BF16> {
  static constexpr int kPerVec = 8;
  static constexpr int kBytes = 2;
  __device__ static __forceinline__ float2 widen(uint32_t w) {
    // bf16 is the upper half of a binary32: widening is a shift.
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  __device__ static __forceinline__ uint32_t narrow(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    uint32_t w;
    memcpy(&w, &h, 4);
    return w;
  }
  __device__ static __forceinline__ float load1(uint64_t a) {
    const unsigned short u = __ldcg(reinterpret_cast<const unsigned short*>(a));
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
  }
  __device__ static __forceinline__ void store1(uint64_t a, float v) {
    *reinterpret_cast<__nv_bfloat16*>(a) = __float2bfloat16_rn(v);
  }
  // Sum of the eight squares of x * k, as for fp32.
  __device__ static __forceinline__ float sumsq(uint4 v, float k) {
    const float2 a = widen(v.x), b = widen(v.y), c = widen(v.z), d = widen(v.w);
    const float y[8] = {__fmul_rn(a.x, k), __fmul_rn(a.y, k), __fmul_rn(b.x, k),
                        __fmul_rn(b.y, k), __fmul_rn(c.x, k), __fmul_rn(c.y, k),
                        __fmul_rn(d.x, k), __fmul_rn(d.y, k)};
    float r = __fmul_rn(y[0], y[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) r = __fmaf_rn(y[i], y[i], r);
    return r;
  }
  __device__ static __forceinline__ uint32_t scale_word(uint32_t w, float chi, float clo) {
    const float2 f = widen(w);
    return narrow(Fmt<GCLIP_F32>::scale1(f.x, chi, clo),
                  Fmt<GCLIP_F32>::scale1(f.y, chi, clo));
  }
  __device__ static __forceinline__ uint4 scale(uint4 v, float chi, float clo) {
    return make_uint4(scale_word(v.x, chi, clo), scale_word(v.y, chi, clo),
                      scale_word(v.z, chi, clo), scale_word(v.w, chi, clo));
  }
  // Element-wise x + a, each sum rounded once to the format: the float sum
  // of two values of a format with p <= 11 significand bits, rounded again
  // to the format, is the correctly rounded sum (24 >= 2p + 2).
  __device__ static __forceinline__ uint32_t add_word(uint32_t x, uint32_t a) {
    const float2 f = widen(x), g = widen(a);
    return narrow(__fadd_rn(f.x, g.x), __fadd_rn(f.y, g.y));
  }
  __device__ static __forceinline__ uint4 add(uint4 x, uint4 a) {
    return make_uint4(add_word(x.x, a.x), add_word(x.y, a.y), add_word(x.z, a.z),
                      add_word(x.w, a.w));
  }
  __device__ static __forceinline__ float round1(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
  }
};

// The elements of one 16-byte vector widened to fp32, element 0 first
// (4 for fp32, 8 for fp16/bf16).
template <int DT>
__device__ __forceinline__ void widen_vec(uint4 g, float (&x)[8]) {
  if constexpr (DT == GCLIP_F32) {
    x[0] = __uint_as_float(g.x);
    x[1] = __uint_as_float(g.y);
    x[2] = __uint_as_float(g.z);
    x[3] = __uint_as_float(g.w);
  } else {
    const float2 a = Fmt<DT>::widen(g.x), b = Fmt<DT>::widen(g.y), c = Fmt<DT>::widen(g.z),
                 d = Fmt<DT>::widen(g.w);
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
    x[4] = c.x; x[5] = c.y; x[6] = d.x; x[7] = d.y;
  }
}

// How one chunk is laid out for vector access: `head` scalar elements up to
// the first 16-byte boundary, `nvec` aligned vectors, then `ntail` scalars.
struct Span {
  uint64_t addr;
  uint64_t body;
  uint32_t head, nvec, tail_start, ntail;
};

template <int DT>
__device__ __forceinline__ Span make_span(uint64_t addr, uint32_t n) {
  constexpr uint32_t E = Fmt<DT>::kPerVec, B = Fmt<DT>::kBytes;
  Span s;
  s.addr = addr;
  s.head = min(n, static_cast<uint32_t>(((16u - (addr & 15u)) & 15u) / B));
  s.body = addr + static_cast<uint64_t>(s.head) * B;
  s.nvec = (n - s.head) / E;
  s.tail_start = s.head + s.nvec * E;
  s.ntail = n - s.tail_start;
  return s;
}

// ---------------------------------------------------------------------------
// Memory access of a chunk's vector body.  Plain: .cg loads for the norm
// pass, streaming (.cs) loads and stores for the scaling pass.  Hinted: the
// same accesses carry an L2 eviction policy made by createpolicy, so that the
// norm pass can keep the chunks it reads last resident in L2 (evict_last)
// for the scaling pass, which visits them first, and let everything else go
// (evict_first).

struct PlainMem {
  __device__ static __forceinline__ uint4 ld_norm(const uint4* p, uint64_t) { return __ldcg(p); }
  __device__ static __forceinline__ uint4 ld_scale(const uint4* p, uint64_t) { return __ldcs(p); }
  __device__ static __forceinline__ void st_scale(uint4* p, uint4 v, uint64_t) { __stcs(p, v); }
};

struct HintMem {
  __device__ static __forceinline__ uint4 ld(const uint4* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
  }
  // Served by L2 even where L1 holds the line: for loads issued before the
  // kernel's own griddepcontrol.wait (k_grad_scale_early).
  __device__ static __forceinline__ uint4 ld_l2(const uint4* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.cg.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
  }
  __device__ static __forceinline__ uint4 ld_norm(const uint4* p, uint64_t pol) { return ld(p, pol); }
  __device__ static __forceinline__ uint4 ld_scale(const uint4* p, uint64_t pol) { return ld(p, pol); }
  __device__ static __forceinline__ void st_scale(uint4* p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;"
                 :
                 : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
  }
};

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

}  // namespace gclip
