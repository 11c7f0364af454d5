// gclip.cu -- global L2-norm gradient clipping for GB300 (sm_103a).
//
// What is computed ("Grow a language model: gradient clipping",
// unhomeschool.com, section "Mathematics"; "Gradient Clipping",
// paweldubiel.com glossary, section "Mechanism and details"):
//     norm = sqrt(sum over every element of every tensor of (x * inv_scale)^2)
//     x <- x * inv_scale * (norm > max_norm ? max_norm / norm : 1)
// with no write at all when that multiplier is exactly 1, and no write and a
// raised flag when an element (or the sum) is not finite.
//
// How.  The clipping page's section "ANDREA's three-kernel pipeline" splits
// the job into a partial-sum kernel (one block per fragment of a tensor,
// results into a small scratch buffer), a final kernel that reduces the
// scratch to one scalar and takes its square root, and a scaling kernel.
// This file keeps that split as one variant and adds a single-launch variant
// in which the last block to finish its partial sums does the final
// reduction and releases the others to scale (the page's heading "Why three
// kernels and not one?" has no body, so the page gives no reason against it).
//
// Both variants share every piece of arithmetic: the per-chunk sum (a fixed
// mapping of elements to the 256 threads of a block, fp32 squares, a
// float-float accumulator, a fixed shuffle tree) and the final reduction (a
// fixed strided order over chunks, the same tree), so the norm and the output
// are bit-identical between variants and from run to run.  The work is a
// streaming reduction bounded by HBM bandwidth; no tensor cores are used.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "internal.hpp"

namespace gclip {

constexpr int kThreads = 256;             // threads per block, every kernel
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 8;                // 16-byte vectors in flight per thread
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
  // Sum of the four squares, one rounding per element (the first product,
  // then fused multiply-adds in element order).
  __device__ static __forceinline__ float sumsq(uint4 v, float s) {
    const float y0 = __fmul_rn(__uint_as_float(v.x), s);
    const float y1 = __fmul_rn(__uint_as_float(v.y), s);
    const float y2 = __fmul_rn(__uint_as_float(v.z), s);
    const float y3 = __fmul_rn(__uint_as_float(v.w), s);
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
  __device__ static __forceinline__ float sumsq(uint4 v, float s) {
    const float2 a = widen(v.x), b = widen(v.y), c = widen(v.z), d = widen(v.w);
    const float y[8] = {__fmul_rn(a.x, s), __fmul_rn(a.y, s), __fmul_rn(b.x, s),
                        __fmul_rn(b.y, s), __fmul_rn(c.x, s), __fmul_rn(c.y, s),
                        __fmul_rn(d.x, s), __fmul_rn(d.y, s)};
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
  __device__ static __forceinline__ float sumsq(uint4 v, float s) {
    const float2 a = widen(v.x), b = widen(v.y), c = widen(v.z), d = widen(v.w);
    const float y[8] = {__fmul_rn(a.x, s), __fmul_rn(a.y, s), __fmul_rn(b.x, s),
                        __fmul_rn(b.y, s), __fmul_rn(c.x, s), __fmul_rn(c.y, s),
                        __fmul_rn(d.x, s), __fmul_rn(d.y, s)};
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
};

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

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// Sum of squares of one chunk: this thread's share, in a fixed order.

template <int DT, class M>
__device__ __forceinline__ FF chunk_sumsq_thread(FF acc, uint64_t addr, uint32_t n, float s,
                                                 uint64_t pol) {
  const Span sp = make_span<DT>(addr, n);
  const uint4* v = reinterpret_cast<const uint4*>(sp.body);
  for (uint32_t base = threadIdx.x; base < sp.nvec; base += kUnroll * kThreads) {
    uint4 buf[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t i = base + u * kThreads;
      buf[u] = i < sp.nvec ? M::ld_norm(v + i, pol) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (base + u * kThreads < sp.nvec) acc = ff_add_f(acc, Fmt<DT>::sumsq(buf[u], s));
    }
  }
  constexpr uint32_t B = Fmt<DT>::kBytes;
  if (threadIdx.x < sp.head) {
    const float y = __fmul_rn(Fmt<DT>::load1(addr + threadIdx.x * B), s);
    acc = ff_add_f(acc, __fmul_rn(y, y));
  }
  if (threadIdx.x < sp.ntail) {
    const float y =
        __fmul_rn(Fmt<DT>::load1(addr + static_cast<uint64_t>(sp.tail_start + threadIdx.x) * B), s);
    acc = ff_add_f(acc, __fmul_rn(y, y));
  }
  return acc;
}

// Fixed-shape tree over the block; the total is valid in thread 0.  `red`
// holds kWarps entries; the trailing barrier lets the caller reuse it.
__device__ __forceinline__ FF block_reduce(FF v, FF* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    FF o;
    o.hi = __shfl_down_sync(0xffffffffu, v.hi, off);
    o.lo = __shfl_down_sync(0xffffffffu, v.lo, off);
    v = ff_add(v, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  FF r = {0.f, 0.f};
  if (warp == 0) {
    r = lane < kWarps ? red[lane] : FF{0.f, 0.f};
#pragma unroll
    for (int off = kWarps / 2; off > 0; off >>= 1) {
      FF o;
      o.hi = __shfl_down_sync(0xffffffffu, r.hi, off);
      o.lo = __shfl_down_sync(0xffffffffu, r.lo, off);
      r = ff_add(r, o);
    }
  }
  __syncthreads();
  return r;
}

// Add this thread's share of chunk `c` to its running accumulator.
template <class M>
__device__ __forceinline__ FF chunk_accumulate(FF acc, const clip_chunk_t& c, float s, uint64_t pol) {
  switch (c.meta & 0xffu) {
    case GCLIP_F32: return chunk_sumsq_thread<GCLIP_F32, M>(acc, c.addr, c.numel, s, pol);
    case GCLIP_F16: return chunk_sumsq_thread<GCLIP_F16, M>(acc, c.addr, c.numel, s, pol);
    default: return chunk_sumsq_thread<GCLIP_BF16, M>(acc, c.addr, c.numel, s, pol);
  }
}

// The sum of squares of one chunk, valid in thread 0.
template <class M>
__device__ __forceinline__ FF chunk_sumsq(const clip_chunk_t& c, float s, FF* red, uint64_t pol) {
  return block_reduce(chunk_accumulate<M>(FF{0.f, 0.f}, c, s, pol), red);
}

// ---------------------------------------------------------------------------
// Scaling of one chunk in place.

template <int DT, class M>
__device__ __forceinline__ void chunk_scale_thread(uint64_t addr, uint32_t n, float chi, float clo,
                                                   uint64_t pol) {
  const Span sp = make_span<DT>(addr, n);
  uint4* v = reinterpret_cast<uint4*>(sp.body);
  for (uint32_t base = threadIdx.x; base < sp.nvec; base += kUnroll * kThreads) {
    uint4 buf[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t i = base + u * kThreads;
      buf[u] = i < sp.nvec ? M::ld_scale(v + i, pol) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t i = base + u * kThreads;
      if (i < sp.nvec) M::st_scale(v + i, Fmt<DT>::scale(buf[u], chi, clo), pol);
    }
  }
  constexpr uint32_t B = Fmt<DT>::kBytes;
  if (threadIdx.x < sp.head) {
    const uint64_t a = addr + threadIdx.x * B;
    Fmt<DT>::store1(a, Fmt<GCLIP_F32>::scale1(Fmt<DT>::load1(a), chi, clo));
  }
  if (threadIdx.x < sp.ntail) {
    const uint64_t a = addr + static_cast<uint64_t>(sp.tail_start + threadIdx.x) * B;
    Fmt<DT>::store1(a, Fmt<GCLIP_F32>::scale1(Fmt<DT>::load1(a), chi, clo));
  }
}

template <class M>
__device__ __forceinline__ void chunk_scale(const clip_chunk_t& c, float chi, float clo, uint64_t pol) {
  switch (c.meta & 0xffu) {
    case GCLIP_F32: chunk_scale_thread<GCLIP_F32, M>(c.addr, c.numel, chi, clo, pol); break;
    case GCLIP_F16: chunk_scale_thread<GCLIP_F16, M>(c.addr, c.numel, chi, clo, pol); break;
    default: chunk_scale_thread<GCLIP_BF16, M>(c.addr, c.numel, chi, clo, pol); break;
  }
}

__device__ __forceinline__ bool must_write(int decision, float chi, float clo) {
  return decision != GCLIP_DECISION_SKIP && !(chi == 1.0f && clo == 0.0f);
}

// ---------------------------------------------------------------------------
// Final reduction over partial sums, square root and decision.  Runs on one
// block of kThreads threads: thread t sums entries t, t + kThreads, ... in
// increasing order, then the fixed block tree; thread 0 writes the record.
//
// The decision is taken in double from the float-float sum: S = hi + lo is
// exact in double, norm = sqrt(S) and max_norm / norm are IEEE double
// operations, and the multiplier inv_scale * max_norm / norm is handed to the
// scaling pass as a float-float pair so that each output is rounded once.

__device__ FF reduce_partials(const float2* partials, int64_t n, FF* red) {
  FF acc = {0.f, 0.f};
  int64_t c = threadIdx.x;
  for (; c + 3 * kThreads < n; c += 4 * kThreads) {
    const float2 p0 = __ldcg(partials + c);
    const float2 p1 = __ldcg(partials + c + kThreads);
    const float2 p2 = __ldcg(partials + c + 2 * kThreads);
    const float2 p3 = __ldcg(partials + c + 3 * kThreads);
    acc = ff_add(acc, FF{p0.x, p0.y});
    acc = ff_add(acc, FF{p1.x, p1.y});
    acc = ff_add(acc, FF{p2.x, p2.y});
    acc = ff_add(acc, FF{p3.x, p3.y});
  }
  for (; c < n; c += kThreads) {
    const float2 p = __ldcg(partials + c);
    acc = ff_add(acc, FF{p.x, p.y});
  }
  return block_reduce(acc, red);
}

// The norm, flag, decision and multiplier from the float-float sum of
// squares S = hi + lo (thread 0).
__device__ void decide_write(FF acc, float max_norm, float inv_scale, clip_result_t* res,
                             float* out_norm, int32_t* out_flag) {
  const double S = static_cast<double>(acc.hi) + static_cast<double>(acc.lo);
  const bool nonfinite = !isfinite(acc.hi) || !isfinite(acc.lo) || S > static_cast<double>(FLT_MAX);
  const double norm = sqrt(S);
  int decision;
  float chi = 1.0f, clo = 0.0f;
  if (nonfinite) {
    decision = GCLIP_DECISION_SKIP;
  } else if (norm > static_cast<double>(max_norm)) {
    decision = GCLIP_DECISION_CLIP;
    const double k = static_cast<double>(inv_scale) * (static_cast<double>(max_norm) / norm);
    chi = __double2float_rn(k);
    clo = __double2float_rn(k - static_cast<double>(chi));
  } else {
    decision = GCLIP_DECISION_PASS;
    chi = inv_scale;
  }
  const float norm_f = __double2float_rn(norm);
  res->norm = norm_f;
  res->nonfinite = nonfinite ? 1 : 0;
  res->decision = decision;
  res->coef_hi = chi;
  res->coef_lo = clo;
  res->sumsq_hi = acc.hi;
  res->sumsq_lo = acc.lo;
  res->calls = res->calls + 1u;
  if (out_norm) *out_norm = norm_f;
  if (out_flag) *out_flag = nonfinite ? 1 : 0;
}

__device__ void final_reduce(const float2* partials, int64_t n_chunks, float max_norm,
                             float inv_scale, clip_result_t* res, float* out_norm,
                             int32_t* out_flag, FF* red) {
  const FF acc = reduce_partials(partials, n_chunks, red);
  if (threadIdx.x == 0) decide_write(acc, max_norm, inv_scale, res, out_norm, out_flag);
}

// ---------------------------------------------------------------------------
// The norm pass of the handle-based clip, shared by both variants.
//
// A grid of G blocks (G fixed per handle: the co-resident count of the
// single-launch kernel, at most the number of chunks).  Block b takes chunks
// b, b + G, b + 2G, ...; each of its threads keeps one float-float
// accumulator over its share of all those chunks, in that order, and the
// block tree combines the threads once at the end.  The block sum goes to
// block_sums[b]; the block that arrives last reduces the G block sums in
// fixed order (final_reduce) and publishes the record.  Which block arrives
// last depends on timing; the arithmetic does not.

struct NormArgs {
  const clip_chunk_t* chunks;
  int64_t n_chunks;
  float2* block_sums;     // G entries
  unsigned int* arrive;   // blocks done with the norm pass in this call
  unsigned int expected;  // G, plus the test hook's extra arrivals
  float max_norm;
  float inv_scale;
  clip_result_t* res;
  float* out_norm;
  int32_t* out_flag;
  int64_t keep_from;      // chunks from here on are read with evict_last
};

__device__ __forceinline__ FF block_norm_pass(const NormArgs& a, FF* red) {
  const uint64_t pol_first = policy_evict_first();
  const uint64_t pol_last = policy_evict_last();
  FF acc = {0.f, 0.f};
  for (int64_t c = blockIdx.x; c < a.n_chunks; c += gridDim.x) {
    const clip_chunk_t ch = a.chunks[c];
    acc = chunk_accumulate<HintMem>(acc, ch, a.inv_scale, c >= a.keep_from ? pol_last : pol_first);
  }
  return block_reduce(acc, red);
}

// Publish this block's sum; returns true (in every thread) in the block that
// arrived last, after it has written the record.
__device__ __forceinline__ bool norm_arrive(const NormArgs& a, FF bsum, FF* red, int* s_flag) {
  if (threadIdx.x == 0) {
    a.block_sums[blockIdx.x] = make_float2(bsum.hi, bsum.lo);
    __threadfence();
    const unsigned int t = atomicAdd(a.arrive, 1u);
    *s_flag = (t + 1u == a.expected);
  }
  __syncthreads();
  if (!*s_flag) return false;
  __threadfence();
  final_reduce(a.block_sums, gridDim.x, a.max_norm, a.inv_scale, a.res, a.out_norm, a.out_flag,
               red);
  if (threadIdx.x == 0) {
    *a.arrive = 0u;  // every block has arrived: rearm for the next call
    __threadfence();
  }
  return true;
}

// ---------------------------------------------------------------------------
// Split variant: the norm pass (with the final reduction in the last block)
// and the scaling pass as two launches.

__global__ void __launch_bounds__(kThreads) k_grad_norm_partial(const NormArgs a) {
  __shared__ FF red[kWarps];
  __shared__ int s_flag;
  // Let the dependent scaling launch be scheduled while this grid runs.
  asm volatile("griddepcontrol.launch_dependents;");
  const FF bsum = block_norm_pass(a, red);
  norm_arrive(a, bsum, red, &s_flag);
}

// One block of the final reduction alone: used when there are no chunks and
// by the no-allocation entry point.
__global__ void __launch_bounds__(kThreads) k_grad_norm_final(const float2* __restrict__ partials,
                                                              int64_t n_chunks, float max_norm,
                                                              float inv_scale, clip_result_t* res,
                                                              float* out_norm, int32_t* out_flag) {
  __shared__ FF red[kWarps];
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  final_reduce(partials, n_chunks, max_norm, inv_scale, res, out_norm, out_flag, red);
}

__global__ void __launch_bounds__(kThreads) k_grad_scale(const clip_chunk_t* __restrict__ chunks,
                                                         int64_t n_chunks,
                                                         const clip_result_t* res) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int decision = res->decision;
  const float chi = res->coef_hi, clo = res->coef_lo;
  if (!must_write(decision, chi, clo)) return;
  // Highest chunks first: the norm pass read them last and kept them in L2.
  const clip_chunk_t c = chunks[n_chunks - 1 - static_cast<int64_t>(blockIdx.x)];
  chunk_scale<HintMem>(c, chi, clo, policy_evict_first());
}

// ---------------------------------------------------------------------------
// Fused clip + AdamW: after the norm pass, one pass over gradients and state
// that forms the clipped gradient in registers and updates w, m, v.

struct TensorState {
  uint64_t g, w, m, v;  // gradient base and the fp32 state arrays of one tensor
};

struct AdamwArgs {
  float beta1, beta2, omb1, omb2;  // beta and 1 - beta, each rounded once to fp32
  float inv_bc1, inv_bc2;          // 1 / (1 - beta^step), from double
  float eps, lr, decay;            // decay = 1 - lr * weight_decay, from double
  int zero_grads;
};

// One element: g^ = x * (chi + clo) rounded once, then the moments and the
// weight, each with IEEE-rounded fp32 operations.
__device__ __forceinline__ void adamw1(float x, float& w, float& m, float& v, float chi, float clo,
                                       const AdamwArgs& p) {
  const float gh = __fmaf_rn(x, chi, __fmul_rn(x, clo));
  m = __fmaf_rn(p.beta1, m, __fmul_rn(p.omb1, gh));
  v = __fmaf_rn(p.beta2, v, __fmul_rn(p.omb2, __fmul_rn(gh, gh)));
  const float denom = __fadd_rn(__fsqrt_rn(__fmul_rn(v, p.inv_bc2)), p.eps);
  const float upd = __fdiv_rn(__fmul_rn(m, p.inv_bc1), denom);
  w = __fmaf_rn(-p.lr, upd, __fmul_rn(w, p.decay));
}

__device__ __forceinline__ void adamw4(const float (&x)[4], float4* w, float4* m, float4* v, float chi,
                                       float clo, const AdamwArgs& p) {
  float4 W = __ldcs(w), M = __ldcs(m), V = __ldcs(v);
  adamw1(x[0], W.x, M.x, V.x, chi, clo, p);
  adamw1(x[1], W.y, M.y, V.y, chi, clo, p);
  adamw1(x[2], W.z, M.z, V.z, chi, clo, p);
  adamw1(x[3], W.w, M.w, V.w, chi, clo, p);
  __stcs(w, W);
  __stcs(m, M);
  __stcs(v, V);
}

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

template <int DT>
__device__ __forceinline__ void adamw_chunk(const clip_chunk_t& c, const TensorState& ts, float chi,
                                            float clo, const AdamwArgs& p) {
  constexpr uint32_t E = Fmt<DT>::kPerVec, B = Fmt<DT>::kBytes;
  const Span sp = make_span<DT>(c.addr, c.numel);
  const uint64_t e0 = (c.addr - ts.g) / B;  // index of the chunk's first element
  float* w = reinterpret_cast<float*>(ts.w) + e0;
  float* m = reinterpret_cast<float*>(ts.m) + e0;
  float* v = reinterpret_cast<float*>(ts.v) + e0;
  const uint64_t pol = policy_evict_first();
  uint4* gv = reinterpret_cast<uint4*>(sp.body);
  const bool vec = ((reinterpret_cast<uint64_t>(w + sp.head) | reinterpret_cast<uint64_t>(m + sp.head) |
                     reinterpret_cast<uint64_t>(v + sp.head)) & 15u) == 0;
  if (vec) {
    for (uint32_t i = threadIdx.x; i < sp.nvec; i += kThreads) {
      float x[8];
      widen_vec<DT>(HintMem::ld_scale(gv + i, pol), x);
      const uint32_t k = sp.head + i * E;
#pragma unroll
      for (uint32_t q = 0; q < E; q += 4) {
        const float xs[4] = {x[q], x[q + 1], x[q + 2], x[q + 3]};
        adamw4(xs, reinterpret_cast<float4*>(w + k + q), reinterpret_cast<float4*>(m + k + q),
               reinterpret_cast<float4*>(v + k + q), chi, clo, p);
      }
      if (p.zero_grads) HintMem::st_scale(gv + i, make_uint4(0, 0, 0, 0), pol);
    }
  } else {
    // state not 16-byte aligned with the gradient: element by element
    for (uint32_t j = sp.head + threadIdx.x; j < sp.tail_start; j += kThreads) {
      const uint64_t a = c.addr + static_cast<uint64_t>(j) * B;
      float W = w[j], M = m[j], V = v[j];
      adamw1(Fmt<DT>::load1(a), W, M, V, chi, clo, p);
      w[j] = W;
      m[j] = M;
      v[j] = V;
      if (p.zero_grads) Fmt<DT>::store1(a, 0.0f);
    }
  }
  for (uint32_t j = threadIdx.x; j < sp.head + sp.ntail; j += kThreads) {
    const uint32_t k = j < sp.head ? j : sp.tail_start + (j - sp.head);
    const uint64_t a = c.addr + static_cast<uint64_t>(k) * B;
    float W = w[k], M = m[k], V = v[k];
    adamw1(Fmt<DT>::load1(a), W, M, V, chi, clo, p);
    w[k] = W;
    m[k] = M;
    v[k] = V;
    if (p.zero_grads) Fmt<DT>::store1(a, 0.0f);
  }
}

__global__ void __launch_bounds__(kThreads) k_adamw(const clip_chunk_t* __restrict__ chunks,
                                                    int64_t n_chunks,
                                                    const TensorState* __restrict__ states,
                                                    const clip_result_t* res, const AdamwArgs p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (__ldcg(&res->decision) == GCLIP_DECISION_SKIP) return;
  const float chi = __ldcg(&res->coef_hi), clo = __ldcg(&res->coef_lo);
  // Highest chunks first: the norm pass read their gradients last.
  const clip_chunk_t c = chunks[n_chunks - 1 - static_cast<int64_t>(blockIdx.x)];
  const TensorState ts = states[c.meta >> 8];
  switch (c.meta & 0xffu) {
    case GCLIP_F32: adamw_chunk<GCLIP_F32>(c, ts, chi, clo, p); break;
    case GCLIP_F16: adamw_chunk<GCLIP_F16>(c, ts, chi, clo, p); break;
    default: adamw_chunk<GCLIP_BF16>(c, ts, chi, clo, p); break;
  }
}

// ---------------------------------------------------------------------------
// Out-of-place clip into fp32: after the norm pass, every element is written
// to its fp32 output as x * (chi + clo), rounded once.

template <int DT>
__device__ __forceinline__ void to_f32_chunk(const clip_chunk_t& c, const TensorState& ts, float chi,
                                             float clo) {
  constexpr uint32_t E = Fmt<DT>::kPerVec, B = Fmt<DT>::kBytes;
  const Span sp = make_span<DT>(c.addr, c.numel);
  const uint64_t e0 = (c.addr - ts.g) / B;
  float* out = reinterpret_cast<float*>(ts.w) + e0;
  const uint64_t pol = policy_evict_first();
  const uint4* gv = reinterpret_cast<const uint4*>(sp.body);
  if ((reinterpret_cast<uint64_t>(out + sp.head) & 15u) == 0) {
    for (uint32_t i = threadIdx.x; i < sp.nvec; i += kThreads) {
      float x[8];
      widen_vec<DT>(HintMem::ld_scale(gv + i, pol), x);
      float4* o = reinterpret_cast<float4*>(out + sp.head + i * E);
#pragma unroll
      for (uint32_t q = 0; q < E; q += 4)
        __stcs(o + q / 4, make_float4(Fmt<GCLIP_F32>::scale1(x[q], chi, clo),
                                      Fmt<GCLIP_F32>::scale1(x[q + 1], chi, clo),
                                      Fmt<GCLIP_F32>::scale1(x[q + 2], chi, clo),
                                      Fmt<GCLIP_F32>::scale1(x[q + 3], chi, clo)));
    }
  } else {
    for (uint32_t j = sp.head + threadIdx.x; j < sp.tail_start; j += kThreads)
      out[j] = Fmt<GCLIP_F32>::scale1(Fmt<DT>::load1(c.addr + static_cast<uint64_t>(j) * B), chi, clo);
  }
  for (uint32_t j = threadIdx.x; j < sp.head + sp.ntail; j += kThreads) {
    const uint32_t k = j < sp.head ? j : sp.tail_start + (j - sp.head);
    out[k] = Fmt<GCLIP_F32>::scale1(Fmt<DT>::load1(c.addr + static_cast<uint64_t>(k) * B), chi, clo);
  }
}

__global__ void __launch_bounds__(kThreads) k_to_f32(const clip_chunk_t* __restrict__ chunks,
                                                     int64_t n_chunks,
                                                     const TensorState* __restrict__ outs,
                                                     const clip_result_t* res) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (__ldcg(&res->decision) == GCLIP_DECISION_SKIP) return;
  const float chi = __ldcg(&res->coef_hi), clo = __ldcg(&res->coef_lo);
  const clip_chunk_t c = chunks[n_chunks - 1 - static_cast<int64_t>(blockIdx.x)];
  const TensorState ts = outs[c.meta >> 8];
  switch (c.meta & 0xffu) {
    case GCLIP_F32: to_f32_chunk<GCLIP_F32>(c, ts, chi, clo); break;
    case GCLIP_F16: to_f32_chunk<GCLIP_F16>(c, ts, chi, clo); break;
    default: to_f32_chunk<GCLIP_BF16>(c, ts, chi, clo); break;
  }
}

// ---------------------------------------------------------------------------
// Per-tensor clipping: each tensor clipped by its own norm.  One block per
// chunk writes the chunk's sum of squares; one block per tensor reduces its
// chunks' sums (the same fixed order as the final reduction) and decides;
// one block per chunk scales with its tensor's multiplier.

__global__ void __launch_bounds__(kThreads) k_chunk_partials(const clip_chunk_t* __restrict__ chunks,
                                                             float inv_scale,
                                                             float2* __restrict__ partials) {
  __shared__ FF red[kWarps];
  asm volatile("griddepcontrol.launch_dependents;");
  const FF acc = chunk_sumsq<HintMem>(chunks[blockIdx.x], inv_scale, red, policy_evict_first());
  if (threadIdx.x == 0) partials[blockIdx.x] = make_float2(acc.hi, acc.lo);
}

__global__ void __launch_bounds__(kThreads) k_tensor_final(const float2* __restrict__ partials,
                                                           const int64_t* __restrict__ first,
                                                           float max_norm, float inv_scale,
                                                           clip_result_t* recs, float* out_norms,
                                                           int32_t* out_flags) {
  __shared__ FF red[kWarps];
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t = blockIdx.x;
  const FF acc = reduce_partials(partials + first[t], first[t + 1] - first[t], red);
  if (threadIdx.x == 0)
    decide_write(acc, max_norm, inv_scale, recs + t, out_norms ? out_norms + t : nullptr,
                 out_flags ? out_flags + t : nullptr);
}

__global__ void __launch_bounds__(kThreads) k_scale_per_tensor(const clip_chunk_t* __restrict__ chunks,
                                                               int64_t n_chunks,
                                                               const clip_result_t* recs) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const clip_chunk_t c = chunks[n_chunks - 1 - static_cast<int64_t>(blockIdx.x)];
  const clip_result_t* r = recs + (c.meta >> 8);
  const int decision = __ldcg(&r->decision);
  const float chi = __ldcg(&r->coef_hi), clo = __ldcg(&r->coef_lo);
  if (!must_write(decision, chi, clo)) return;
  chunk_scale<HintMem>(c, chi, clo, policy_evict_first());
}

// ---------------------------------------------------------------------------
// Single-launch variant (cooperative launch, so every block is resident).

__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__global__ void __launch_bounds__(kThreads, 5) k_clip_persistent(const NormArgs a, SyncWords* sync,
                                                              long long timeout_ns) {
  __shared__ FF red[kWarps];
  __shared__ unsigned int s_gen0, s_claim;
  __shared__ int s_flag, s_go;

  // The generation before this call.  It is bumped only after every block
  // has arrived, so each block reads the same value here.
  if (threadIdx.x == 0) s_gen0 = *reinterpret_cast<volatile unsigned int*>(&sync->gen);

  // Phase 1: the norm pass; the block that arrives last publishes the record.
  const FF bsum = block_norm_pass(a, red);
  const bool published = norm_arrive(a, bsum, red, &s_flag);

  if (published) {
    if (threadIdx.x == 0) {
      sync->work = 0u;  // nobody claims before the generation moves
      __threadfence();
      atomicAdd(&sync->gen, 1u);  // release: the record was fenced above
      s_go = 1;
    }
  } else if (threadIdx.x == 0) {
    // Bounded wait for the record; on timeout flag it and write nothing.
    const unsigned long long t0 = globaltimer();
    int ok = 1;
    while (ld_acquire(&sync->gen) == s_gen0) {
      if (static_cast<long long>(globaltimer() - t0) > timeout_ns) {
        atomicExch(&a.res->status, GCLIP_STATUS_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
    s_go = ok;
  }
  __syncthreads();
  if (!s_go) return;

  const int decision = __ldcg(&a.res->decision);
  const float chi = __ldcg(&a.res->coef_hi), clo = __ldcg(&a.res->coef_lo);
  if (!must_write(decision, chi, clo)) return;
  // Phase 2: chunks claimed one at a time from a shared counter, highest
  // chunk first (most recently read).  Thread 0 claims the next chunk while
  // the block scales the current one.
  const uint64_t pol = policy_evict_first();
  const unsigned int n = static_cast<unsigned int>(a.n_chunks);
  if (threadIdx.x == 0) s_claim = atomicAdd(&sync->work, 1u);
  __syncthreads();
  unsigned int claim = s_claim;
  while (claim < n) {
    unsigned int next = 0;
    if (threadIdx.x == 0) next = atomicAdd(&sync->work, 1u);
    chunk_scale<HintMem>(a.chunks[n - 1u - claim], chi, clo, pol);
    __syncthreads();
    if (threadIdx.x == 0) s_claim = next;
    __syncthreads();
    claim = s_claim;
  }
}

// ===========================================================================
// TMA engine: the same two passes with bulk copies through a ring of shared
// memory stages.  Two blocks per SM; each block's issuing thread keeps up to
// kStages chunk bodies (the 16-byte-aligned run of each chunk, at most
// GCLIP_CHUNK_BYTES) in flight with cp.async.bulk, each stage completing on
// its own mbarrier; all 256 threads consume a stage from shared memory with
// the same element-to-thread mapping as the register engine.  The scaling
// pass rewrites the stage in shared memory and stores it back with a bulk
// store.  Every wait is bounded: on timeout the block records
// GCLIP_STATUS_TIMEOUT, waits (bounded) for the copies it still has in
// flight, and returns without writing gradients.

constexpr int kStages = 3;
constexpr uint32_t kStageBytes = GCLIP_CHUNK_BYTES;
constexpr size_t kTmaSmem = static_cast<size_t>(kStages) * kStageBytes + kStages * sizeof(uint64_t);
constexpr long long kRingTimeoutNs = 1000000000LL;  // one chunk copy: 1 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on one phase, by thread 0 alone; true if it completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long timeout_ns) {
  const unsigned long long t0 = globaltimer();
  uint32_t spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++spins & 255u) == 0 && static_cast<long long>(globaltimer() - t0) > timeout_ns) return false;
  }
  return true;
}

__device__ __forceinline__ void bulk_load(void* dst, uint64_t src, uint32_t bytes, uint64_t* bar,
                                          uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void bulk_store(uint64_t dst, const void* src, uint32_t bytes, uint64_t pol) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
               "r"(smem_addr(src)), "r"(bytes), "l"(pol)
               : "memory");
}

// Close this thread's bulk-store group (possibly empty), one per chunk.
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Bulk stores of this thread: at most N groups may still be reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The aligned vector body of a chunk: device address and byte count.
__device__ __forceinline__ void chunk_body(const clip_chunk_t& c, uint64_t& addr, uint32_t& bytes) {
  const uint32_t es = (c.meta & 0xffu) == GCLIP_F32 ? 4u : 2u;
  const uint32_t per = 16u / es;
  const uint32_t head = min(c.numel, static_cast<uint32_t>(((16u - (c.addr & 15u)) & 15u) / es));
  addr = c.addr + static_cast<uint64_t>(head) * es;
  bytes = (c.numel - head) / per * 16u;
}

// Thread 0: start the copy of chunk `c` into stage `st`.
__device__ __forceinline__ void ring_issue(uint8_t* st, uint64_t* bar, const clip_chunk_t& c, uint64_t pol) {
  uint64_t src;
  uint32_t bytes;
  chunk_body(c, src, bytes);
  if (bytes) {
    mbar_expect_tx(bar, bytes);
    bulk_load(st, src, bytes, bar, pol);
  } else {
    mbar_arrive(bar);
  }
}

// The ring's shared memory: kStages data stages, then kStages mbarriers.
struct Ring {
  uint8_t* data;
  uint64_t* full;
  __device__ uint8_t* stage(int s) const { return data + static_cast<size_t>(s) * kStageBytes; }
};

__device__ __forceinline__ Ring ring_setup(uint8_t* smem) {
  Ring r;
  r.data = smem;
  r.full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(kStages) * kStageBytes);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&r.full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  return r;
}

// Stage k % kStages holds the k-th chunk of this block's sequence; `phase`
// keeps, per stage, the parity of its next phase.  Every thread keeps the
// same copy and flips a bit for each chunk it consumes.
__device__ __forceinline__ uint32_t take_parity(uint32_t& phase, int s) {
  const uint32_t p = (phase >> s) & 1u;
  phase ^= 1u << s;
  return p;
}

// Thread 0: wait, bounded, for the copies of chunks k .. issued - 1.
__device__ __forceinline__ void ring_drain(const Ring& r, int64_t k, int64_t issued, uint32_t phase,
                                           long long timeout_ns) {
  for (int64_t j = k; j < issued; ++j) {
    const int s = static_cast<int>(j % kStages);
    mbar_wait_bounded(&r.full[s], take_parity(phase, s), timeout_ns);
  }
}

// Wait for chunk k to land.  Every thread waits for itself (the wait also
// makes the stage's contents visible to it).  A thread that gives up records
// the status and raises the block's abort flag, which the block reads after
// its next barrier.
__device__ __forceinline__ bool ring_wait(const Ring& r, int64_t k, uint32_t& phase, clip_result_t* res,
                                          volatile int* s_abort) {
  const int s = static_cast<int>(k % kStages);
  const uint32_t parity = take_parity(phase, s);
  if (mbar_wait_bounded(&r.full[s], parity, kRingTimeoutNs)) return true;
  atomicExch(&res->status, GCLIP_STATUS_TIMEOUT);
  *s_abort = 1;
  return false;
}

// After the barrier that follows chunk k: if any thread gave up, thread 0
// waits (bounded) for the copies that may still be in flight, chunk k's
// included, and the block returns.  `phase` is thread 0's, already advanced
// past chunk k, so chunk k's bit is turned back first.
__device__ __forceinline__ bool ring_aborted(const Ring& r, int64_t k, int64_t issued, uint32_t phase,
                                             volatile int* s_abort) {
  if (!*s_abort) return false;
  if (threadIdx.x == 0)
    ring_drain(r, k, issued, phase ^ (1u << static_cast<int>(k % kStages)), kRingTimeoutNs / 10);
  return true;
}

// This thread's share of one staged chunk, added to four independent
// accumulators (vector j of the thread's share goes to acc[j % 4]) so that
// four float-float chains run side by side; head and tail scalars go to
// acc[0].  The order is fixed, so the result is deterministic.
template <int DT>
__device__ __forceinline__ void stage_sumsq(FF (&acc)[4], const uint8_t* st, const clip_chunk_t& c,
                                            float s) {
  const Span sp = make_span<DT>(c.addr, c.numel);
  const uint4* v = reinterpret_cast<const uint4*>(st);
  uint32_t i = threadIdx.x;
  for (; i + 3 * kThreads < sp.nvec; i += 4 * kThreads) {
    const uint4 v0 = v[i], v1 = v[i + kThreads], v2 = v[i + 2 * kThreads], v3 = v[i + 3 * kThreads];
    acc[0] = ff_add_f(acc[0], Fmt<DT>::sumsq(v0, s));
    acc[1] = ff_add_f(acc[1], Fmt<DT>::sumsq(v1, s));
    acc[2] = ff_add_f(acc[2], Fmt<DT>::sumsq(v2, s));
    acc[3] = ff_add_f(acc[3], Fmt<DT>::sumsq(v3, s));
  }
  // fewer than four vectors left: constant indices keep acc in registers
  if (i < sp.nvec) acc[0] = ff_add_f(acc[0], Fmt<DT>::sumsq(v[i], s));
  if (i + kThreads < sp.nvec) acc[1] = ff_add_f(acc[1], Fmt<DT>::sumsq(v[i + kThreads], s));
  if (i + 2 * kThreads < sp.nvec) acc[2] = ff_add_f(acc[2], Fmt<DT>::sumsq(v[i + 2 * kThreads], s));
  constexpr uint32_t B = Fmt<DT>::kBytes;
  if (threadIdx.x < sp.head) {
    const float y = __fmul_rn(Fmt<DT>::load1(c.addr + threadIdx.x * B), s);
    acc[0] = ff_add_f(acc[0], __fmul_rn(y, y));
  }
  if (threadIdx.x < sp.ntail) {
    const float y =
        __fmul_rn(Fmt<DT>::load1(c.addr + static_cast<uint64_t>(sp.tail_start + threadIdx.x) * B), s);
    acc[0] = ff_add_f(acc[0], __fmul_rn(y, y));
  }
}

template <int DT>
__device__ __forceinline__ void stage_scale(uint8_t* st, const clip_chunk_t& c, float chi, float clo) {
  const Span sp = make_span<DT>(c.addr, c.numel);
  uint4* v = reinterpret_cast<uint4*>(st);
  for (uint32_t i = threadIdx.x; i < sp.nvec; i += kThreads) v[i] = Fmt<DT>::scale(v[i], chi, clo);
  constexpr uint32_t B = Fmt<DT>::kBytes;
  if (threadIdx.x < sp.head) {
    const uint64_t a = c.addr + threadIdx.x * B;
    Fmt<DT>::store1(a, Fmt<GCLIP_F32>::scale1(Fmt<DT>::load1(a), chi, clo));
  }
  if (threadIdx.x < sp.ntail) {
    const uint64_t a = c.addr + static_cast<uint64_t>(sp.tail_start + threadIdx.x) * B;
    Fmt<DT>::store1(a, Fmt<GCLIP_F32>::scale1(Fmt<DT>::load1(a), chi, clo));
  }
}

// Chunk k of this block's sequence in the norm pass (increasing) and in the
// scaling pass (decreasing, most recently read first).
__device__ __forceinline__ int64_t norm_chunk(int64_t k) { return blockIdx.x + k * gridDim.x; }
__device__ __forceinline__ int64_t scale_chunk(int64_t n, int64_t k) {
  return n - 1 - (blockIdx.x + k * gridDim.x);
}
__device__ __forceinline__ int64_t my_count(int64_t n) {
  return blockIdx.x < n ? (n - 1 - blockIdx.x) / gridDim.x + 1 : 0;
}

// Norm pass through the ring; the block sum is valid in thread 0.  Returns
// false (uniformly) if a copy timed out; no copy is then in flight.
__device__ bool tma_norm_pass(const NormArgs& a, const Ring& r, uint32_t& phase, FF* red,
                              volatile int* s_abort, FF* out) {
  const int64_t mine = my_count(a.n_chunks);
  const uint64_t pol_first = policy_evict_first(), pol_last = policy_evict_last();
  int64_t issued = 0;
  if (threadIdx.x == 0) {
    for (; issued < kStages && issued < mine; ++issued) {
      const int64_t c = norm_chunk(issued);
      ring_issue(r.stage(static_cast<int>(issued)), &r.full[issued], a.chunks[c],
                 c >= a.keep_from ? pol_last : pol_first);
    }
  }
  FF acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
  for (int64_t k = 0; k < mine; ++k) {
    const int s = static_cast<int>(k % kStages);
    if (ring_wait(r, k, phase, a.res, s_abort)) {
      const clip_chunk_t ch = a.chunks[norm_chunk(k)];
      switch (ch.meta & 0xffu) {
        case GCLIP_F32: stage_sumsq<GCLIP_F32>(acc, r.stage(s), ch, a.inv_scale); break;
        case GCLIP_F16: stage_sumsq<GCLIP_F16>(acc, r.stage(s), ch, a.inv_scale); break;
        default: stage_sumsq<GCLIP_BF16>(acc, r.stage(s), ch, a.inv_scale); break;
      }
    }
    __syncthreads();
    if (ring_aborted(r, k, issued, phase, s_abort)) return false;
    if (threadIdx.x == 0 && issued < mine) {
      const int64_t c = norm_chunk(issued);
      fence_proxy_async();
      ring_issue(r.stage(s), &r.full[s], a.chunks[c], c >= a.keep_from ? pol_last : pol_first);
      ++issued;
    }
  }
  *out = block_reduce(ff_add(ff_add(acc[0], acc[1]), ff_add(acc[2], acc[3])), red);
  return true;
}

// Thread 0: prefetch the first kStages - 1 chunks of the scaling pass.
__device__ __forceinline__ int64_t tma_scale_prefetch(const clip_chunk_t* chunks, int64_t n, const Ring& r,
                                                      uint64_t pol) {
  const int64_t mine = my_count(n);
  int64_t issued = 0;
  fence_proxy_async();
  for (; issued < kStages - 1 && issued < mine; ++issued)
    ring_issue(r.stage(static_cast<int>(issued)), &r.full[issued], chunks[scale_chunk(n, issued)], pol);
  return issued;
}

// Scaling pass through the ring, after tma_scale_prefetch (thread 0's
// `issued` counts the chunks it has started).  Returns false (uniformly) if a
// copy timed out; no copy or store is then in flight.
__device__ bool tma_scale_pass(const clip_chunk_t* chunks, int64_t n, const Ring& r, uint32_t& phase,
                               int64_t issued, float chi, float clo, clip_result_t* res,
                               volatile int* s_abort) {
  const int64_t mine = my_count(n);
  const uint64_t pol = policy_evict_first();
  for (int64_t k = 0; k < mine; ++k) {
    const int s = static_cast<int>(k % kStages);
    const clip_chunk_t ch = chunks[scale_chunk(n, k)];
    if (ring_wait(r, k, phase, res, s_abort)) {
      switch (ch.meta & 0xffu) {
        case GCLIP_F32: stage_scale<GCLIP_F32>(r.stage(s), ch, chi, clo); break;
        case GCLIP_F16: stage_scale<GCLIP_F16>(r.stage(s), ch, chi, clo); break;
        default: stage_scale<GCLIP_BF16>(r.stage(s), ch, chi, clo); break;
      }
    }
    fence_proxy_async();  // this thread's shared-memory writes, visible to the bulk store
    __syncthreads();
    if (ring_aborted(r, k, issued, phase, s_abort)) {
      if (threadIdx.x == 0) bulk_wait_all();
      return false;
    }
    if (threadIdx.x == 0) {
      uint64_t dst;
      uint32_t bytes;
      chunk_body(ch, dst, bytes);
      if (bytes) bulk_store(dst, r.stage(s), bytes, pol);
      bulk_commit();
      if (issued < mine) {
        // The stage of chunk `issued` last held chunk k - 1, whose store
        // group was committed one iteration ago: wait until at most the
        // newest group (chunk k's) is still reading shared memory.
        bulk_wait_read<1>();
        const int ns = static_cast<int>(issued % kStages);
        ring_issue(r.stage(ns), &r.full[ns], chunks[scale_chunk(n, issued)], pol);
        ++issued;
      }
    }
  }
  if (threadIdx.x == 0) bulk_wait_all();
  return true;
}

__global__ void __launch_bounds__(kThreads, 2) k_norm_tma(const NormArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ FF red[kWarps];
  __shared__ int s_abort, s_flag;
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) s_abort = 0;
  const Ring r = ring_setup(smem);
  uint32_t phase = 0;
  FF bsum;
  // A block whose copy timed out still arrives, with a NaN sum, so that the
  // record is published and says SKIP.
  if (!tma_norm_pass(a, r, phase, red, &s_abort, &bsum) && threadIdx.x == 0)
    bsum = FF{__int_as_float(0x7fc00000), 0.f};
  norm_arrive(a, bsum, red, &s_flag);
}

__global__ void __launch_bounds__(kThreads, 2) k_scale_tma(const clip_chunk_t* __restrict__ chunks, int64_t n,
                                                           clip_result_t* res) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_abort, s_go;
  if (threadIdx.x == 0) s_abort = 0;
  const Ring r = ring_setup(smem);
  uint32_t phase = 0;
  // The gradients are not written by the norm pass, so the first chunks can
  // be fetched before the record exists; they are most likely in L2.
  int64_t issued = 0;
  if (threadIdx.x == 0) issued = tma_scale_prefetch(chunks, n, r, policy_evict_first());
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int decision = __ldcg(&res->decision);
  const float chi = __ldcg(&res->coef_hi), clo = __ldcg(&res->coef_lo);
  if (threadIdx.x == 0) s_go = must_write(decision, chi, clo) ? 1 : 0;
  __syncthreads();
  if (!s_go) {
    // Nothing to write: let the prefetched copies land before leaving.
    if (threadIdx.x == 0) ring_drain(r, 0, issued, phase, kRingTimeoutNs);
    return;
  }
  tma_scale_pass(chunks, n, r, phase, issued, chi, clo, res, &s_abort);
}

__global__ void __launch_bounds__(kThreads, 2) k_clip_persistent_tma(const NormArgs a, SyncWords* sync,
                                                                     long long timeout_ns) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ FF red[kWarps];
  __shared__ unsigned int s_gen0;
  __shared__ int s_abort, s_flag, s_go;
  if (threadIdx.x == 0) {
    s_gen0 = *reinterpret_cast<volatile unsigned int*>(&sync->gen);
    s_abort = 0;
  }
  const Ring r = ring_setup(smem);
  uint32_t phase = 0;
  FF bsum;
  const bool ok = tma_norm_pass(a, r, phase, red, &s_abort, &bsum);
  // A block whose copy timed out still arrives, with a NaN sum (so the clip
  // is skipped), to keep the others from waiting for it.
  if (!ok && threadIdx.x == 0) bsum = FF{__int_as_float(0x7fc00000), 0.f};
  const bool published = norm_arrive(a, bsum, red, &s_flag);

  // Speculative prefetch of the scaling pass while the record is pending.
  int64_t issued = 0;
  if (threadIdx.x == 0 && ok) issued = tma_scale_prefetch(a.chunks, a.n_chunks, r, policy_evict_first());

  if (published) {
    if (threadIdx.x == 0) {
      atomicAdd(&sync->gen, 1u);
      s_go = 1;
    }
  } else if (threadIdx.x == 0) {
    const unsigned long long t0 = globaltimer();
    unsigned int ns = 32;
    int go = 1;
    while (ld_acquire(&sync->gen) == s_gen0) {
      if (static_cast<long long>(globaltimer() - t0) > timeout_ns) {
        atomicExch(&a.res->status, GCLIP_STATUS_TIMEOUT);
        go = 0;
        break;
      }
      __nanosleep(ns);
      if (ns < 1024) ns <<= 1;
    }
    __threadfence();
    s_go = go;
  }
  __syncthreads();
  const int decision = __ldcg(&a.res->decision);
  const float chi = __ldcg(&a.res->coef_hi), clo = __ldcg(&a.res->coef_lo);
  if (!ok || !s_go || !must_write(decision, chi, clo)) {
    if (threadIdx.x == 0) ring_drain(r, 0, issued, phase, kRingTimeoutNs);
    return;
  }
  tma_scale_pass(a.chunks, a.n_chunks, r, phase, issued, chi, clo, a.res, &s_abort);
}

}  // namespace gclip

// ===========================================================================
// Host side: the C ABI.

using gclip::SyncWords;

struct gclip_handle {
  int device;
  int64_t n_chunks;
  int64_t keep_from;         // first chunk the norm pass reads with evict_last
  int64_t l2_bytes;          // L2 size of the device
  int32_t variant;
  int32_t grid_persistent;   // blocks of the register engine (co-resident)
  int32_t grid_tma;          // blocks of the TMA engine (co-resident)
  int32_t coop;
  int32_t debug_extra;
  long long timeout_ns;
  void* arena;
  clip_chunk_t* d_chunks;
  float2* d_partials;        // one entry per block of the norm pass (G)
  clip_result_t* d_result;
  SyncWords* d_sync;
  int64_t* d_first;          // first chunk of each tensor, n_tensors + 1 entries
  clip_result_t* d_trec;     // per-tensor records of clip_grad_norm_per_tensor
  std::vector<clip_tensor_desc_t> descs;   // the gradient tensors, as created
  gclip::TensorState* d_states;            // AdamW state table (NULL until attached)
  gclip::TensorState* d_outs;              // fp32 output table (NULL until attached)
};

namespace {

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Make the handle's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
      return;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

bool valid_scalar(float v) { return std::isfinite(v) && v > 0.0f; }

// The norm pass marks its last `bytes` (rounded to whole chunks) evict_last
// in L2, for the scaling pass to find there.
void set_keep(gclip_handle* h, int64_t bytes) {
  const int64_t k = bytes / GCLIP_CHUNK_BYTES;
  h->keep_from = k >= h->n_chunks ? 0 : h->n_chunks - k;
}

gclip::NormArgs norm_args(gclip_handle* h, int32_t grid, float max_norm, float inv_scale,
                          float* out_norm, int32_t* out_flag, unsigned int extra) {
  gclip::NormArgs a;
  a.chunks = h->d_chunks;
  a.n_chunks = h->n_chunks;
  a.block_sums = h->d_partials;
  a.arrive = &h->d_sync->arrive;
  a.expected = static_cast<unsigned int>(grid) + extra;
  a.max_norm = max_norm;
  a.inv_scale = inv_scale;
  a.res = h->d_result;
  a.out_norm = out_norm;
  a.out_flag = out_flag;
  a.keep_from = h->keep_from;
  return a;
}

cudaError_t launch_pdl(const void* fn, unsigned int grid, cudaStream_t s, void** args, bool pdl,
                       size_t smem = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(gclip::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

extern "C" int clip_create(const clip_tensor_desc_t* descs, int32_t n_tensors, clip_handle_t* out) {
  if (out == nullptr) return GCLIP_ERR_INVALID_ARG;
  std::vector<clip_chunk_t> chunks;
  int rc = gclip::build_chunks(descs, n_tensors, chunks);
  if (rc != GCLIP_OK) return rc;

  gclip_handle* h = new (std::nothrow) gclip_handle();
  if (h == nullptr) return GCLIP_ERR_OOM;
  if (cudaGetDevice(&h->device) != cudaSuccess) {
    delete h;
    return GCLIP_ERR_CUDA;
  }
  h->n_chunks = static_cast<int64_t>(chunks.size());
  h->variant = GCLIP_VARIANT_SPLIT;
  h->descs.assign(descs, descs + n_tensors);
  h->timeout_ns = gclip::kDefaultTimeoutNs;

  const size_t n = chunks.size();
  // G, the norm pass's grid, is known only after the occupancy query below;
  // it is at most the number of chunks, so size the block sums for that.
  const size_t off_chunks = 0;
  const size_t off_partials = round_up(off_chunks + n * sizeof(clip_chunk_t), 256);
  const size_t off_result = round_up(off_partials + n * sizeof(float2), 256);
  const size_t off_sync = round_up(off_result + sizeof(clip_result_t), 256);
  const size_t nt = static_cast<size_t>(n_tensors);
  const size_t off_first = round_up(off_sync + sizeof(SyncWords), 256);
  const size_t off_trec = round_up(off_first + (nt + 1) * sizeof(int64_t), 256);
  const size_t total = round_up(off_trec + (nt ? nt : 1) * sizeof(clip_result_t), 256);
  std::vector<int64_t> first(nt + 1, 0);
  {
    size_t c = 0;
    for (size_t t = 0; t < nt; ++t) {
      first[t] = static_cast<int64_t>(c);
      while (c < n && (chunks[c].meta >> 8) == t) ++c;
    }
    first[nt] = static_cast<int64_t>(c);
  }
  cudaError_t e = cudaMalloc(&h->arena, total);
  if (e != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return e == cudaErrorMemoryAllocation ? GCLIP_ERR_OOM : GCLIP_ERR_CUDA;
  }
  char* base = static_cast<char*>(h->arena);
  h->d_chunks = reinterpret_cast<clip_chunk_t*>(base + off_chunks);
  h->d_partials = reinterpret_cast<float2*>(base + off_partials);
  h->d_result = reinterpret_cast<clip_result_t*>(base + off_result);
  h->d_sync = reinterpret_cast<SyncWords*>(base + off_sync);
  h->d_first = reinterpret_cast<int64_t*>(base + off_first);
  h->d_trec = reinterpret_cast<clip_result_t*>(base + off_trec);

  int sms = 0, per_sm = 0, coop = 0, l2 = 0;
  e = cudaMemset(h->arena, 0, total);
  if (e == cudaSuccess && n > 0)
    e = cudaMemcpy(h->d_chunks, chunks.data(), n * sizeof(clip_chunk_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(h->d_first, first.data(), first.size() * sizeof(int64_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, h->device);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gclip::k_clip_persistent,
                                                      gclip::kThreads, 0);
  int per_sm_tma = 0;
  for (const void* fn : {reinterpret_cast<const void*>(gclip::k_norm_tma),
                         reinterpret_cast<const void*>(gclip::k_scale_tma),
                         reinterpret_cast<const void*>(gclip::k_clip_persistent_tma)})
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(gclip::kTmaSmem));
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_tma, gclip::k_clip_persistent_tma,
                                                      gclip::kThreads, gclip::kTmaSmem);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->arena);
    delete h;
    return GCLIP_ERR_CUDA;
  }
  h->l2_bytes = l2;
  set_keep(h, 0);
  const int64_t resident = static_cast<int64_t>(sms) * per_sm;
  h->grid_persistent = static_cast<int32_t>(resident < h->n_chunks ? resident : h->n_chunks);
  const int64_t resident_tma = static_cast<int64_t>(sms) * per_sm_tma;
  h->grid_tma = static_cast<int32_t>(resident_tma < h->n_chunks ? resident_tma : h->n_chunks);
  h->coop = coop;
  *out = h;
  return GCLIP_OK;
}

namespace {

// Enqueue one clip.  `events` (may be NULL) are recorded between the steps;
// programmatic dependent launch is used only when no events are recorded.
int enqueue(clip_handle_t h, float max_norm, float inv_scale, float* out_norm,
            int32_t* out_flag, cudaStream_t s, cudaEvent_t const* events) {
  int64_t nc = h->n_chunks;
  const float2* partials = h->d_partials;
  const bool pdl = events == nullptr;
  cudaError_t e = cudaSuccess;
  auto mark = [&](int i) {
    if (events != nullptr && e == cudaSuccess) e = cudaEventRecord(events[i], s);
  };

  mark(0);
  if (nc == 0) {
    mark(1);
    mark(2);
    void* args[] = {&partials, &nc, &max_norm, &inv_scale, &h->d_result, &out_norm, &out_flag};
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_final), 1, s, args, false);
  } else if (h->variant == GCLIP_VARIANT_SPLIT) {
    gclip::NormArgs a = norm_args(h, h->grid_persistent, max_norm, inv_scale, out_norm, out_flag, 0);
    void* a1[] = {&a};
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_partial),
                     static_cast<unsigned int>(h->grid_persistent), s, a1, false);
    mark(1);
    mark(2);
    const clip_chunk_t* chunks = h->d_chunks;
    const clip_result_t* cres = h->d_result;
    void* a3[] = {&chunks, &nc, &cres};
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_scale),
                     static_cast<unsigned int>(nc), s, a3, pdl);
  } else if (h->variant == GCLIP_VARIANT_SPLIT_TMA) {
    gclip::NormArgs a = norm_args(h, h->grid_tma, max_norm, inv_scale, out_norm, out_flag, 0);
    void* a1[] = {&a};
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_norm_tma),
                     static_cast<unsigned int>(h->grid_tma), s, a1, false, gclip::kTmaSmem);
    mark(1);
    mark(2);
    const clip_chunk_t* chunks = h->d_chunks;
    clip_result_t* res = h->d_result;
    void* a3[] = {&chunks, &nc, &res};
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_scale_tma),
                     static_cast<unsigned int>(h->grid_tma), s, a3, pdl, gclip::kTmaSmem);
  } else if (h->variant == GCLIP_VARIANT_PERSISTENT_TMA) {
    mark(1);
    mark(2);
    gclip::NormArgs a = norm_args(h, h->grid_tma, max_norm, inv_scale, out_norm, out_flag,
                                  static_cast<unsigned int>(h->debug_extra));
    long long tmo = h->timeout_ns;
    if (e == cudaSuccess && h->debug_extra > 0)
      e = cudaMemsetAsync(h->d_sync, 0, sizeof(SyncWords), s);
    if (e == cudaSuccess) {
      SyncWords* sync = h->d_sync;
      void* args[] = {&a, &sync, &tmo};
      e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(gclip::k_clip_persistent_tma),
                                      dim3(h->grid_tma), dim3(gclip::kThreads), args, gclip::kTmaSmem,
                                      s);
    }
    if (e == cudaSuccess && h->debug_extra > 0)
      e = cudaMemsetAsync(h->d_sync, 0, sizeof(SyncWords), s);
  } else {
    mark(1);
    mark(2);
    gclip::NormArgs a = norm_args(h, h->grid_persistent, max_norm, inv_scale, out_norm, out_flag,
                                  static_cast<unsigned int>(h->debug_extra));
    long long tmo = h->timeout_ns;
    if (e == cudaSuccess && h->debug_extra > 0)
      e = cudaMemsetAsync(h->d_sync, 0, sizeof(SyncWords), s);
    if (e == cudaSuccess) {
      SyncWords* sync = h->d_sync;
      void* args[] = {&a, &sync, &tmo};
      e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(gclip::k_clip_persistent),
                                      dim3(h->grid_persistent), dim3(gclip::kThreads), args, 0, s);
    }
    if (e == cudaSuccess && h->debug_extra > 0)
      e = cudaMemsetAsync(h->d_sync, 0, sizeof(SyncWords), s);
  }
  mark(3);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GCLIP_ERR_CUDA;
  }
  return GCLIP_OK;
}

}  // namespace

extern "C" int clip_grad_norm(clip_handle_t h, float max_norm, float inv_scale, float* out_norm,
                              int32_t* out_nonfinite_flag, void* stream) {
  if (h == nullptr || !valid_scalar(max_norm) || !valid_scalar(inv_scale))
    return GCLIP_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok) return GCLIP_ERR_CUDA;
  return enqueue(h, max_norm, inv_scale, out_norm, out_nonfinite_flag,
                 static_cast<cudaStream_t>(stream), nullptr);
}

extern "C" int clip_grad_norm_profiled(clip_handle_t h, float max_norm, float inv_scale,
                                       float* out_norm, int32_t* out_nonfinite_flag, void* stream,
                                       void* const* events) {
  if (h == nullptr || events == nullptr || !valid_scalar(max_norm) || !valid_scalar(inv_scale))
    return GCLIP_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i)
    if (events[i] == nullptr) return GCLIP_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok) return GCLIP_ERR_CUDA;
  return enqueue(h, max_norm, inv_scale, out_norm, out_nonfinite_flag,
                 static_cast<cudaStream_t>(stream), reinterpret_cast<cudaEvent_t const*>(events));
}

extern "C" int clip_destroy(clip_handle_t h) {
  if (h == nullptr) return GCLIP_OK;
  int rc = GCLIP_OK;
  {
    DeviceGuard guard(h->device);
    if (!guard.ok || cudaDeviceSynchronize() != cudaSuccess) rc = GCLIP_ERR_CUDA;
    if (cudaFree(h->arena) != cudaSuccess) rc = GCLIP_ERR_CUDA;
    if (h->d_states != nullptr && cudaFree(h->d_states) != cudaSuccess) rc = GCLIP_ERR_CUDA;
    if (h->d_outs != nullptr && cudaFree(h->d_outs) != cudaSuccess) rc = GCLIP_ERR_CUDA;
    cudaGetLastError();
  }
  delete h;
  return rc;
}

extern "C" int clip_set_variant(clip_handle_t h, int32_t variant) {
  if (h == nullptr) return GCLIP_ERR_INVALID_ARG;
  if (variant < GCLIP_VARIANT_SPLIT || variant > GCLIP_VARIANT_PERSISTENT_TMA)
    return GCLIP_ERR_INVALID_ARG;
  const bool coop = variant == GCLIP_VARIANT_PERSISTENT || variant == GCLIP_VARIANT_PERSISTENT_TMA;
  const int32_t grid = (variant == GCLIP_VARIANT_SPLIT_TMA || variant == GCLIP_VARIANT_PERSISTENT_TMA)
                           ? h->grid_tma
                           : h->grid_persistent;
  if ((coop && !h->coop) || (grid <= 0 && h->n_chunks > 0)) return GCLIP_ERR_UNSUPPORTED;
  h->variant = variant;
  return GCLIP_OK;
}

extern "C" int32_t clip_get_variant(clip_handle_t h) { return h ? h->variant : -1; }

extern "C" const clip_result_t* clip_result_device(clip_handle_t h) {
  return h ? h->d_result : nullptr;
}

extern "C" int clip_read_result(clip_handle_t h, clip_result_t* out, void* stream) {
  if (h == nullptr || out == nullptr) return GCLIP_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok) return GCLIP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(out, h->d_result, sizeof(clip_result_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GCLIP_ERR_CUDA;
  }
  return GCLIP_OK;
}

extern "C" int clip_reset(clip_handle_t h, void* stream) {
  if (h == nullptr) return GCLIP_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok) return GCLIP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(h->d_sync, 0, sizeof(SyncWords), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(&h->d_result->status, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GCLIP_ERR_CUDA;
  }
  return GCLIP_OK;
}

extern "C" int64_t clip_num_chunks(clip_handle_t h) { return h ? h->n_chunks : -1; }

extern "C" int32_t clip_persistent_grid(clip_handle_t h) { return h ? h->grid_persistent : -1; }

extern "C" int32_t clip_tma_grid(clip_handle_t h) { return h ? h->grid_tma : -1; }

extern "C" int clip_set_l2_keep(clip_handle_t h, int64_t bytes) {
  if (h == nullptr || bytes < 0) return GCLIP_ERR_INVALID_ARG;
  set_keep(h, bytes);
  return GCLIP_OK;
}

extern "C" int clip_debug_barrier(clip_handle_t h, int32_t extra_arrivals, int64_t timeout_ns) {
  if (h == nullptr || extra_arrivals < 0 || timeout_ns < 0) return GCLIP_ERR_INVALID_ARG;
  h->debug_extra = extra_arrivals;
  h->timeout_ns = timeout_ns > 0 ? timeout_ns : gclip::kDefaultTimeoutNs;
  return GCLIP_OK;
}

namespace {

// Validate per-tensor fp32 arrays (`per` of them for each tensor, `ptrs`
// laid out tensor by tensor) against the handle's gradients, and replace
// *slot with a device table of {gradient base, arrays...}.
int attach_table(clip_handle_t h, const float* const* ptrs, int per, int32_t n_tensors,
                 gclip::TensorState** slot) {
  if (h == nullptr || n_tensors != static_cast<int32_t>(h->descs.size()) ||
      (n_tensors > 0 && ptrs == nullptr))
    return GCLIP_ERR_INVALID_ARG;
  std::vector<clip_tensor_desc_t> all(h->descs);  // gradients, then every array
  std::vector<gclip::TensorState> table(static_cast<size_t>(n_tensors));
  for (int32_t t = 0; t < n_tensors; ++t) {
    const clip_tensor_desc_t& d = h->descs[t];
    uint64_t* f = &table[t].w;
    table[t].g = reinterpret_cast<uint64_t>(d.ptr);
    table[t].w = table[t].m = table[t].v = 0;
    for (int k = 0; k < per; ++k) {
      const float* a = ptrs[static_cast<size_t>(t) * per + k];
      f[k] = reinterpret_cast<uint64_t>(a);
      if (d.numel == 0) continue;
      clip_tensor_desc_t s = {const_cast<float*>(a), d.numel, GCLIP_F32, 0};
      all.push_back(s);
    }
  }
  if (gclip::validate_descs(all.data(), static_cast<int32_t>(all.size())) != GCLIP_OK)
    return GCLIP_ERR_INVALID_ARG;  // NULL, misaligned or overlapping
  DeviceGuard guard(h->device);
  if (!guard.ok) return GCLIP_ERR_CUDA;
  gclip::TensorState* d = nullptr;
  const size_t bytes = sizeof(gclip::TensorState) * (table.empty() ? 1 : table.size());
  cudaError_t e = cudaMalloc(&d, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? GCLIP_ERR_OOM : GCLIP_ERR_CUDA;
  }
  if (!table.empty())
    e = cudaMemcpy(d, table.data(), table.size() * sizeof(gclip::TensorState),
                   cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaGetLastError();
    cudaFree(d);
    return GCLIP_ERR_CUDA;
  }
  if (*slot != nullptr) {
    cudaDeviceSynchronize();  // the old table may still be read by queued work
    cudaFree(*slot);
  }
  *slot = d;
  return GCLIP_OK;
}

// The split norm pass followed by one per-chunk kernel `fn` launched with
// programmatic dependent launch on `args` (after the norm pass's own).
int enqueue_norm_then(clip_handle_t h, float max_norm, float inv_scale, float* out_norm,
                      int32_t* out_flag, cudaStream_t s, const void* fn, void** args) {
  int64_t nc = h->n_chunks;
  cudaError_t e = cudaSuccess;
  if (nc == 0) {
    const float2* partials = h->d_partials;
    void* a[] = {&partials, &nc, &max_norm, &inv_scale, &h->d_result, &out_norm, &out_flag};
    e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_final), 1, s, a, false);
  } else {
    gclip::NormArgs a = norm_args(h, h->grid_persistent, max_norm, inv_scale, out_norm, out_flag, 0);
    void* a1[] = {&a};
    e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_partial),
                   static_cast<unsigned int>(h->grid_persistent), s, a1, false);
    if (e == cudaSuccess) e = launch_pdl(fn, static_cast<unsigned int>(nc), s, args, true);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GCLIP_ERR_CUDA;
  }
  return GCLIP_OK;
}

}  // namespace

extern "C" int clip_attach_adamw(clip_handle_t h, const clip_adamw_state_t* states,
                                 int32_t n_tensors) {
  if (h == nullptr || (n_tensors > 0 && states == nullptr)) return GCLIP_ERR_INVALID_ARG;
  std::vector<const float*> ptrs;
  for (int32_t t = 0; t < n_tensors; ++t) {
    ptrs.push_back(states[t].w);
    ptrs.push_back(states[t].m);
    ptrs.push_back(states[t].v);
  }
  return attach_table(h, ptrs.data(), 3, n_tensors, &h->d_states);
}

extern "C" int clip_attach_f32_out(clip_handle_t h, float* const* outs, int32_t n_tensors) {
  if (h == nullptr) return GCLIP_ERR_INVALID_ARG;
  return attach_table(h, const_cast<const float* const*>(outs), 1, n_tensors, &h->d_outs);
}

extern "C" int clip_grad_norm_to_f32(clip_handle_t h, float max_norm, float inv_scale,
                                     float* out_norm, int32_t* out_nonfinite_flag, void* stream) {
  if (h == nullptr || h->d_outs == nullptr || !valid_scalar(max_norm) || !valid_scalar(inv_scale))
    return GCLIP_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok) return GCLIP_ERR_CUDA;
  int64_t nc = h->n_chunks;
  const clip_chunk_t* chunks = h->d_chunks;
  const gclip::TensorState* outs = h->d_outs;
  const clip_result_t* cres = h->d_result;
  void* args[] = {&chunks, &nc, &outs, &cres};
  return enqueue_norm_then(h, max_norm, inv_scale, out_norm, out_nonfinite_flag,
                           static_cast<cudaStream_t>(stream),
                           reinterpret_cast<const void*>(gclip::k_to_f32), args);
}

extern "C" int clip_grad_norm_adamw(clip_handle_t h, float max_norm, float inv_scale,
                                    const clip_adamw_params_t* p, int64_t step, float* out_norm,
                                    int32_t* out_nonfinite_flag, void* stream) {
  if (h == nullptr || p == nullptr || h->d_states == nullptr || !valid_scalar(max_norm) ||
      !valid_scalar(inv_scale) || step < 1)
    return GCLIP_ERR_INVALID_ARG;
  const bool ok = std::isfinite(p->lr) && p->lr >= 0.0f && std::isfinite(p->eps) && p->eps > 0.0f &&
                  std::isfinite(p->weight_decay) && p->weight_decay >= 0.0f && p->beta1 >= 0.0f &&
                  p->beta1 < 1.0f && p->beta2 >= 0.0f && p->beta2 < 1.0f;
  if (!ok) return GCLIP_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok) return GCLIP_ERR_CUDA;
  gclip::AdamwArgs q;
  const double b1 = p->beta1, b2 = p->beta2;
  q.beta1 = p->beta1;
  q.beta2 = p->beta2;
  q.omb1 = static_cast<float>(1.0 - b1);
  q.omb2 = static_cast<float>(1.0 - b2);
  q.inv_bc1 = static_cast<float>(1.0 / (1.0 - std::pow(b1, static_cast<double>(step))));
  q.inv_bc2 = static_cast<float>(1.0 / (1.0 - std::pow(b2, static_cast<double>(step))));
  q.eps = p->eps;
  q.lr = p->lr;
  q.decay = static_cast<float>(1.0 - static_cast<double>(p->lr) * p->weight_decay);
  q.zero_grads = p->zero_grads ? 1 : 0;
  int64_t nc = h->n_chunks;
  const clip_chunk_t* chunks = h->d_chunks;
  const gclip::TensorState* st = h->d_states;
  const clip_result_t* cres = h->d_result;
  void* args[] = {&chunks, &nc, &st, &cres, &q};
  return enqueue_norm_then(h, max_norm, inv_scale, out_norm, out_nonfinite_flag,
                           static_cast<cudaStream_t>(stream),
                           reinterpret_cast<const void*>(gclip::k_adamw), args);
}

extern "C" int clip_grad_norm_per_tensor(clip_handle_t h, float max_norm, float inv_scale,
                                         float* out_norms, int32_t* out_nonfinite_flags,
                                         void* stream) {
  if (h == nullptr || !valid_scalar(max_norm) || !valid_scalar(inv_scale))
    return GCLIP_ERR_INVALID_ARG;
  const unsigned int nt = static_cast<unsigned int>(h->descs.size());
  if (nt == 0) return GCLIP_OK;
  DeviceGuard guard(h->device);
  if (!guard.ok) return GCLIP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int64_t nc = h->n_chunks;
  const clip_chunk_t* chunks = h->d_chunks;
  float2* partials = h->d_partials;
  const float2* cpartials = partials;
  const int64_t* first = h->d_first;
  clip_result_t* recs = h->d_trec;
  const clip_result_t* crecs = recs;
  cudaError_t e = cudaSuccess;
  if (nc > 0) {
    void* a1[] = {&chunks, &inv_scale, &partials};
    e = launch_pdl(reinterpret_cast<const void*>(gclip::k_chunk_partials),
                   static_cast<unsigned int>(nc), s, a1, false);
  }
  void* a2[] = {&cpartials, &first, &max_norm, &inv_scale, &recs, &out_norms, &out_nonfinite_flags};
  if (e == cudaSuccess)
    e = launch_pdl(reinterpret_cast<const void*>(gclip::k_tensor_final), nt, s, a2, nc > 0);
  void* a3[] = {&chunks, &nc, &crecs};
  if (e == cudaSuccess && nc > 0)
    e = launch_pdl(reinterpret_cast<const void*>(gclip::k_scale_per_tensor),
                   static_cast<unsigned int>(nc), s, a3, true);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GCLIP_ERR_CUDA;
  }
  return GCLIP_OK;
}

extern "C" int clip_read_per_tensor(clip_handle_t h, clip_result_t* out, int32_t n, void* stream) {
  if (h == nullptr || out == nullptr || n < 0 || n > static_cast<int32_t>(h->descs.size()))
    return GCLIP_ERR_INVALID_ARG;
  if (n == 0) return GCLIP_OK;
  DeviceGuard guard(h->device);
  if (!guard.ok) return GCLIP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(out, h->d_trec, sizeof(clip_result_t) * n, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GCLIP_ERR_CUDA;
  }
  return GCLIP_OK;
}

// ===========================================================================
// No-allocation entry point: one contiguous buffer, scratch in a fixed array.

namespace gclip {

// The scratch of clip_grad_norm_flat_noalloc: the per-chunk partial sums,
// then the result record.  Compiled into the library, so it costs every GPU
// that loads the library GCLIP_NOALLOC_SCRATCH_BYTES until exit.
constexpr size_t kNoAllocPartialBytes = static_cast<size_t>(GCLIP_NOALLOC_MAX_CHUNKS) * 8;
static_assert(kNoAllocPartialBytes + sizeof(clip_result_t) <= GCLIP_NOALLOC_SCRATCH_BYTES,
              "record does not fit the scratch");
static __device__ __align__(256) unsigned char g_noalloc_scratch[GCLIP_NOALLOC_SCRATCH_BYTES];

// Chunk c of a single tensor at `base`, cut exactly as the host planner cuts
// one tensor: the first chunk takes the elements before the first 16-byte
// boundary plus a full chunk, every later chunk starts aligned.
__device__ __forceinline__ clip_chunk_t flat_chunk(uint64_t base, int64_t numel, int32_t dtype,
                                                   int64_t c) {
  const int64_t es = dtype == GCLIP_F32 ? 4 : 2;
  const int64_t per = GCLIP_CHUNK_BYTES / es;
  const int64_t head = static_cast<int64_t>((16u - (base & 15u)) & 15u) / es;
  const int64_t start = c == 0 ? 0 : head + c * per;
  const int64_t want = c == 0 ? head + per : per;
  const int64_t left = numel - start;
  clip_chunk_t ch;
  ch.addr = base + static_cast<uint64_t>(start * es);
  ch.numel = static_cast<uint32_t>(left < want ? left : want);
  ch.meta = static_cast<uint32_t>(dtype);
  return ch;
}

__global__ void __launch_bounds__(kThreads) k_grad_norm_partial_flat(uint64_t base, int64_t numel,
                                                                     int32_t dtype, float inv_scale,
                                                                     float2* __restrict__ partials) {
  __shared__ FF red[kWarps];
  asm volatile("griddepcontrol.launch_dependents;");
  const clip_chunk_t c = flat_chunk(base, numel, dtype, blockIdx.x);
  const FF acc = chunk_sumsq<PlainMem>(c, inv_scale, red, 0);
  if (threadIdx.x == 0) partials[blockIdx.x] = make_float2(acc.hi, acc.lo);
}

__global__ void __launch_bounds__(kThreads) k_grad_scale_flat(uint64_t base, int64_t numel,
                                                              int32_t dtype, int64_t n_chunks,
                                                              const clip_result_t* res) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int decision = res->decision;
  const float chi = res->coef_hi, clo = res->coef_lo;
  if (!must_write(decision, chi, clo)) return;
  const clip_chunk_t c =
      flat_chunk(base, numel, dtype, n_chunks - 1 - static_cast<int64_t>(blockIdx.x));
  chunk_scale<PlainMem>(c, chi, clo, 0);
}

}  // namespace gclip

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoAllocMaxDevices];  // device address of the scratch, per device

// Device address of the scratch array on `dev` (current), looked up once.
void* noalloc_scratch(int dev) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, gclip::g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_noalloc_addr[dev] = p;
  }
  return g_noalloc_addr[dev];
}

}  // namespace

extern "C" int clip_grad_norm_flat_noalloc(void* grads, int64_t numel, int32_t dtype,
                                           float max_norm, float inv_scale, float* out_norm,
                                           int32_t* out_nonfinite_flag, void* stream) {
  const int es = gclip::elem_size(dtype);
  if (es == 0 || numel < 0 || !valid_scalar(max_norm) || !valid_scalar(inv_scale))
    return GCLIP_ERR_INVALID_ARG;
  const uint64_t base = reinterpret_cast<uint64_t>(grads);
  if (numel > 0 && (base == 0 || base % static_cast<uint64_t>(es) != 0))
    return GCLIP_ERR_INVALID_ARG;
  const int64_t per = GCLIP_CHUNK_BYTES / es;
  const int64_t head = static_cast<int64_t>((16u - (base & 15u)) & 15u) / es;
  // The first chunk holds head + per elements, every other chunk per.
  if (numel > head + static_cast<int64_t>(GCLIP_NOALLOC_MAX_CHUNKS) * per)
    return GCLIP_ERR_TOO_LARGE;
  int64_t nc = 0;
  if (numel > 0) nc = numel <= head + per ? 1 : 1 + (numel - head - 1) / per;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GCLIP_ERR_CUDA;
  }
  char* scratch = static_cast<char*>(noalloc_scratch(dev));
  if (scratch == nullptr) return GCLIP_ERR_CUDA;
  float2* partials = reinterpret_cast<float2*>(scratch);
  clip_result_t* record = reinterpret_cast<clip_result_t*>(scratch + gclip::kNoAllocPartialBytes);
  const float2* cpartials = partials;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;

  void* a2[] = {&cpartials, &nc, &max_norm, &inv_scale, &record, &out_norm, &out_nonfinite_flag};
  if (nc == 0) {
    e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_final), 1, s, a2, false);
  } else {
    uint64_t b = base;
    int64_t n = numel;
    int32_t dt = dtype;
    void* a1[] = {&b, &n, &dt, &inv_scale, &partials};
    e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_partial_flat),
                   static_cast<unsigned int>(nc), s, a1, false);
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_final), 1, s, a2, true);
    const clip_result_t* crecord = record;
    void* a3[] = {&b, &n, &dt, &nc, &crecord};
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_scale_flat),
                     static_cast<unsigned int>(nc), s, a3, true);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GCLIP_ERR_CUDA;
  }
  return GCLIP_OK;
}
