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
  unsigned int arrive;  // blocks that finished their partial sums this call
  unsigned int gen;     // bumped once per call when the record is published
  unsigned int pad[2];
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
// Sum of squares of one chunk: this thread's share, in a fixed order.

template <int DT>
__device__ __forceinline__ FF chunk_sumsq_thread(uint64_t addr, uint32_t n, float s) {
  const Span sp = make_span<DT>(addr, n);
  const uint4* v = reinterpret_cast<const uint4*>(sp.body);
  FF acc = {0.f, 0.f};
  for (uint32_t base = threadIdx.x; base < sp.nvec; base += kUnroll * kThreads) {
    uint4 buf[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t i = base + u * kThreads;
      buf[u] = i < sp.nvec ? __ldcg(v + i) : make_uint4(0, 0, 0, 0);
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

__device__ __forceinline__ FF chunk_sumsq(const clip_chunk_t& c, float s, FF* red) {
  FF acc;
  switch (c.meta & 0xffu) {
    case GCLIP_F32: acc = chunk_sumsq_thread<GCLIP_F32>(c.addr, c.numel, s); break;
    case GCLIP_F16: acc = chunk_sumsq_thread<GCLIP_F16>(c.addr, c.numel, s); break;
    default: acc = chunk_sumsq_thread<GCLIP_BF16>(c.addr, c.numel, s); break;
  }
  return block_reduce(acc, red);
}

// ---------------------------------------------------------------------------
// Scaling of one chunk in place.  Loads and stores are marked streaming
// (evict-first): this data is not read again.

template <int DT>
__device__ __forceinline__ void chunk_scale_thread(uint64_t addr, uint32_t n, float chi, float clo) {
  const Span sp = make_span<DT>(addr, n);
  uint4* v = reinterpret_cast<uint4*>(sp.body);
  for (uint32_t base = threadIdx.x; base < sp.nvec; base += kUnroll * kThreads) {
    uint4 buf[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t i = base + u * kThreads;
      buf[u] = i < sp.nvec ? __ldcs(v + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t i = base + u * kThreads;
      if (i < sp.nvec) __stcs(v + i, Fmt<DT>::scale(buf[u], chi, clo));
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

__device__ __forceinline__ void chunk_scale(const clip_chunk_t& c, float chi, float clo) {
  switch (c.meta & 0xffu) {
    case GCLIP_F32: chunk_scale_thread<GCLIP_F32>(c.addr, c.numel, chi, clo); break;
    case GCLIP_F16: chunk_scale_thread<GCLIP_F16>(c.addr, c.numel, chi, clo); break;
    default: chunk_scale_thread<GCLIP_BF16>(c.addr, c.numel, chi, clo); break;
  }
}

__device__ __forceinline__ bool must_write(int decision, float chi, float clo) {
  return decision != GCLIP_DECISION_SKIP && !(chi == 1.0f && clo == 0.0f);
}

// ---------------------------------------------------------------------------
// Final reduction over the per-chunk partial sums, square root and decision.
// Runs on one block of kThreads threads; the record is written by thread 0.
//
// The decision is taken in double from the float-float sum: S = hi + lo is
// exact in double, norm = sqrt(S) and max_norm / norm are IEEE double
// operations, and the multiplier inv_scale * max_norm / norm is handed to the
// scaling pass as a float-float pair so that each output is rounded once.

__device__ void final_reduce(const float2* partials, int64_t n_chunks, float max_norm,
                             float inv_scale, clip_result_t* res, float* out_norm,
                             int32_t* out_flag, FF* red) {
  FF acc = {0.f, 0.f};
  int64_t c = threadIdx.x;
  for (; c + 3 * kThreads < n_chunks; c += 4 * kThreads) {
    const float2 p0 = __ldcg(partials + c);
    const float2 p1 = __ldcg(partials + c + kThreads);
    const float2 p2 = __ldcg(partials + c + 2 * kThreads);
    const float2 p3 = __ldcg(partials + c + 3 * kThreads);
    acc = ff_add(acc, FF{p0.x, p0.y});
    acc = ff_add(acc, FF{p1.x, p1.y});
    acc = ff_add(acc, FF{p2.x, p2.y});
    acc = ff_add(acc, FF{p3.x, p3.y});
  }
  for (; c < n_chunks; c += kThreads) {
    const float2 p = __ldcg(partials + c);
    acc = ff_add(acc, FF{p.x, p.y});
  }
  acc = block_reduce(acc, red);
  if (threadIdx.x != 0) return;

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

// ---------------------------------------------------------------------------
// Three-kernel variant.

__global__ void __launch_bounds__(kThreads) k_grad_norm_partial(const clip_chunk_t* __restrict__ chunks,
                                                                float inv_scale,
                                                                float2* __restrict__ partials) {
  __shared__ FF red[kWarps];
  // Let the dependent final-reduce launch be scheduled while this grid runs.
  asm volatile("griddepcontrol.launch_dependents;");
  const clip_chunk_t c = chunks[blockIdx.x];
  const FF acc = chunk_sumsq(c, inv_scale, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = make_float2(acc.hi, acc.lo);
}

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
  // Highest chunks first: the partial pass read them last, so they are the
  // ones most likely still held in L2.
  const clip_chunk_t c = chunks[n_chunks - 1 - static_cast<int64_t>(blockIdx.x)];
  chunk_scale(c, chi, clo);
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

__global__ void __launch_bounds__(kThreads) k_clip_persistent(
    const clip_chunk_t* __restrict__ chunks, int64_t n_chunks, float max_norm, float inv_scale,
    float2* __restrict__ partials, clip_result_t* res, float* out_norm, int32_t* out_flag,
    SyncWords* sync, unsigned int expected, long long timeout_ns) {
  __shared__ FF red[kWarps];
  __shared__ unsigned int s_gen0;
  __shared__ int s_last, s_go;

  // The generation before this call; it changes only after every block has
  // arrived, so each block reads the same value here.
  if (threadIdx.x == 0) s_gen0 = *reinterpret_cast<volatile unsigned int*>(&sync->gen);

  // Phase 1: per-chunk partial sums, chunks strided over the grid.
  for (int64_t c = blockIdx.x; c < n_chunks; c += gridDim.x) {
    const clip_chunk_t ch = chunks[c];
    const FF acc = chunk_sumsq(ch, inv_scale, red);
    if (threadIdx.x == 0) partials[c] = make_float2(acc.hi, acc.lo);
  }

  // Arrival: the block that takes the last ticket reduces.
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int t = atomicAdd(&sync->arrive, 1u);
    s_last = (t + 1u == expected);
  }
  __syncthreads();

  if (s_last) {
    __threadfence();
    final_reduce(partials, n_chunks, max_norm, inv_scale, res, out_norm, out_flag, red);
    __syncthreads();
    if (threadIdx.x == 0) {
      sync->arrive = 0u;  // every block has arrived: safe to rearm
      __threadfence();
      atomicAdd(&sync->gen, 1u);
      s_go = 1;
    }
  } else if (threadIdx.x == 0) {
    // Bounded wait for the record; on timeout flag it and write nothing.
    const unsigned long long t0 = globaltimer();
    unsigned int ns = 32;
    int ok = 1;
    while (ld_acquire(&sync->gen) == s_gen0) {
      if (static_cast<long long>(globaltimer() - t0) > timeout_ns) {
        atomicExch(&res->status, GCLIP_STATUS_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(ns);
      if (ns < 1024) ns <<= 1;
    }
    __threadfence();
    s_go = ok;
  }
  __syncthreads();
  if (!s_go) return;

  const int decision = __ldcg(&res->decision);
  const float chi = __ldcg(&res->coef_hi), clo = __ldcg(&res->coef_lo);
  if (!must_write(decision, chi, clo)) return;
  // Phase 2: the same chunks in reverse order, most recently read first.
  for (int64_t k = blockIdx.x; k < n_chunks; k += gridDim.x) {
    const clip_chunk_t ch = chunks[n_chunks - 1 - k];
    chunk_scale(ch, chi, clo);
  }
}

}  // namespace gclip

// ===========================================================================
// Host side: the C ABI.

using gclip::SyncWords;

struct gclip_handle {
  int device;
  int64_t n_chunks;
  int32_t variant;
  int32_t grid_persistent;
  int32_t coop;
  int32_t debug_extra;
  long long timeout_ns;
  void* arena;
  clip_chunk_t* d_chunks;
  float2* d_partials;
  clip_result_t* d_result;
  SyncWords* d_sync;
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

cudaError_t launch_pdl(const void* fn, unsigned int grid, cudaStream_t s, void** args, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(gclip::kThreads);
  cfg.dynamicSmemBytes = 0;
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
  h->variant = GCLIP_VARIANT_THREE_KERNEL;
  h->timeout_ns = gclip::kDefaultTimeoutNs;

  const size_t n = chunks.size();
  const size_t off_chunks = 0;
  const size_t off_partials = round_up(off_chunks + n * sizeof(clip_chunk_t), 256);
  const size_t off_result = round_up(off_partials + n * sizeof(float2), 256);
  const size_t off_sync = round_up(off_result + sizeof(clip_result_t), 256);
  const size_t total = round_up(off_sync + sizeof(SyncWords), 256);
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

  int sms = 0, per_sm = 0, coop = 0;
  e = cudaMemset(h->arena, 0, total);
  if (e == cudaSuccess && n > 0)
    e = cudaMemcpy(h->d_chunks, chunks.data(), n * sizeof(clip_chunk_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->device);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gclip::k_clip_persistent,
                                                      gclip::kThreads, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->arena);
    delete h;
    return GCLIP_ERR_CUDA;
  }
  const int64_t resident = static_cast<int64_t>(sms) * per_sm;
  h->grid_persistent = static_cast<int32_t>(resident < h->n_chunks ? resident : h->n_chunks);
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
    void* args[] = {&partials, &nc, &max_norm, &inv_scale, &h->d_result, &out_norm, &out_flag};
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_final), 1, s, args, false);
    mark(2);
  } else if (h->variant == GCLIP_VARIANT_THREE_KERNEL) {
    const clip_chunk_t* chunks = h->d_chunks;
    float2* wpartials = h->d_partials;
    void* a1[] = {&chunks, &inv_scale, &wpartials};
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_partial),
                     static_cast<unsigned int>(nc), s, a1, false);
    mark(1);
    void* a2[] = {&partials, &nc, &max_norm, &inv_scale, &h->d_result, &out_norm, &out_flag};
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_final), 1, s, a2, pdl);
    mark(2);
    const clip_result_t* cres = h->d_result;
    void* a3[] = {&chunks, &nc, &cres};
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_scale),
                     static_cast<unsigned int>(nc), s, a3, pdl);
  } else {
    mark(1);
    mark(2);
    const clip_chunk_t* chunks = h->d_chunks;
    float2* wpartials = h->d_partials;
    unsigned int expected =
        static_cast<unsigned int>(h->grid_persistent) + static_cast<unsigned int>(h->debug_extra);
    long long tmo = h->timeout_ns;
    if (e == cudaSuccess && h->debug_extra > 0)
      e = cudaMemsetAsync(h->d_sync, 0, sizeof(SyncWords), s);
    if (e == cudaSuccess) {
      void* args[] = {&chunks,   &nc,       &max_norm,   &inv_scale, &wpartials, &h->d_result,
                      &out_norm, &out_flag, &h->d_sync,  &expected,  &tmo};
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
    cudaGetLastError();
  }
  delete h;
  return rc;
}

extern "C" int clip_set_variant(clip_handle_t h, int32_t variant) {
  if (h == nullptr) return GCLIP_ERR_INVALID_ARG;
  if (variant != GCLIP_VARIANT_THREE_KERNEL && variant != GCLIP_VARIANT_PERSISTENT)
    return GCLIP_ERR_INVALID_ARG;
  if (variant == GCLIP_VARIANT_PERSISTENT && (!h->coop || (h->grid_persistent <= 0 && h->n_chunks > 0)))
    return GCLIP_ERR_UNSUPPORTED;
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

extern "C" int clip_debug_barrier(clip_handle_t h, int32_t extra_arrivals, int64_t timeout_ns) {
  if (h == nullptr || extra_arrivals < 0 || timeout_ns < 0) return GCLIP_ERR_INVALID_ARG;
  h->debug_extra = extra_arrivals;
  h->timeout_ns = timeout_ns > 0 ? timeout_ns : gclip::kDefaultTimeoutNs;
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
  const FF acc = chunk_sumsq(c, inv_scale, red);
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
  chunk_scale(c, chi, clo);
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
