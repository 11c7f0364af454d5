// reduce.cuh -- the arithmetic of the norm: per-thread sums of squares of a
// chunk (plain, or with the last microbatch added in), the fixed block tree,
// the scaling of a chunk, the final reduction with the decision in
// float-float (double when the tiny bin is not empty),
// and the norm pass shared by the register-engine variants.
// Included by gclip.cu only.
#pragma once

#include <cfloat>

#include "common.cuh"

namespace gclip {

// ---------------------------------------------------------------------------
// Squares of one vector or one element into the two bins (see SumSq).  The
// vector's sum r of the squares of y = x * s (the first square, then fused
// multiply-adds in element order) goes to `big` unless r < kTinySq; such a
// vector is summed again as the squares of x * st (st = s * 2^K) into
// `tiny`.  r < 2^-100 means every |y| < 2^-50, and r >= 2^-100 means the
// squares that underflowed (each off by at most 2^-150) change r by less
// than 2^-46 of itself.  A NaN or infinite r goes to `big`.  The common case
// costs one comparison and a branch that is not taken.

template <int DT>
__device__ __forceinline__ void vec_sumsq(FF& big, FF& tiny, uint4 v, float s, float st) {
  const float r = Fmt<DT>::sumsq(v, s);
  if (__builtin_expect(r < kTinySq, 0)) tiny = ff_add_f(tiny, Fmt<DT>::sumsq(v, st));
  else big = ff_add_f(big, r);
}

template <int DT>
__device__ __forceinline__ void vec_sumsq(SumSq& acc, uint4 v, float s, float st) {
  vec_sumsq<DT>(acc.big, acc.tiny, v, s, st);
}

__device__ __forceinline__ void elem_sumsq(FF& big, FF& tiny, float x, float s, float st) {
  const float y = __fmul_rn(x, s);
  const float r = __fmul_rn(y, y);
  if (__builtin_expect(r < kTinySq, 0)) {
    const float z = __fmul_rn(x, st);
    tiny = ff_add_f(tiny, __fmul_rn(z, z));
  } else {
    big = ff_add_f(big, r);
  }
}

__device__ __forceinline__ void elem_sumsq(SumSq& acc, float x, float s, float st) {
  elem_sumsq(acc.big, acc.tiny, x, s, st);
}

// ---------------------------------------------------------------------------
// Sum of squares of one chunk: this thread's share, in a fixed order.

template <int DT, class M>
__device__ __forceinline__ void chunk_sumsq_thread(SumSq& acc, uint64_t addr, uint32_t n, float s,
                                                   float st, uint64_t pol) {
  const Span sp = make_span<DT>(addr, n);
  const uint4* v = reinterpret_cast<const uint4*>(sp.body);
  for (uint32_t base = threadIdx.x; base < sp.nvec; base += kNormUnroll * kThreads) {
    uint4 buf[kNormUnroll];
#pragma unroll
    for (int u = 0; u < kNormUnroll; ++u) {
      const uint32_t i = base + u * kThreads;
      buf[u] = i < sp.nvec ? M::ld_norm(v + i, pol) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kNormUnroll; ++u) {
      if (base + u * kThreads < sp.nvec) vec_sumsq<DT>(acc, buf[u], s, st);
    }
  }
  constexpr uint32_t B = Fmt<DT>::kBytes;
  if (threadIdx.x < sp.head) elem_sumsq(acc, Fmt<DT>::load1(addr + threadIdx.x * B), s, st);
  if (threadIdx.x < sp.ntail)
    elem_sumsq(acc, Fmt<DT>::load1(addr + static_cast<uint64_t>(sp.tail_start + threadIdx.x) * B), s,
               st);
}

// Fixed-shape tree over the block; the total is valid in thread 0.  `red`
// holds kWarps entries; the trailing barrier lets the caller reuse it.
__device__ __forceinline__ FF warp_reduce(FF v, int width) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    if (off >= width) continue;
    FF o;
    o.hi = __shfl_down_sync(0xffffffffu, v.hi, off);
    o.lo = __shfl_down_sync(0xffffffffu, v.lo, off);
    v = ff_add(v, o);
  }
  return v;
}

// The tiny bin is usually +0 in every thread (it only ever adds squares):
// a warp whose tiny bins are all +0 skips their tree, whose result would be
// +0 anyway.
__device__ __forceinline__ bool any_tiny(const FF& t) {
  return __any_sync(0xffffffffu, t.hi != 0.f || t.lo != 0.f);
}

__device__ __forceinline__ SumSq block_reduce(SumSq v, SumSq* red) {
  v.big = warp_reduce(v.big, 32);
  if (any_tiny(v.tiny)) v.tiny = warp_reduce(v.tiny, 32);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  SumSq r = {{0.f, 0.f}, {0.f, 0.f}};
  if (warp == 0) {
    if (lane < kWarps) r = red[lane];
    r.big = warp_reduce(r.big, kWarps);
    if (any_tiny(r.tiny)) r.tiny = warp_reduce(r.tiny, kWarps);
  }
  __syncthreads();
  return r;
}

// Add this thread's share of chunk `c` to its running accumulator.
template <class M>
__device__ __forceinline__ void chunk_accumulate(SumSq& acc, const clip_chunk_t& c, float s, float st,
                                                 uint64_t pol) {
  switch (c.meta & 0xffu) {
    case GCLIP_F32: chunk_sumsq_thread<GCLIP_F32, M>(acc, c.addr, c.numel, s, st, pol); break;
    case GCLIP_F16: chunk_sumsq_thread<GCLIP_F16, M>(acc, c.addr, c.numel, s, st, pol); break;
    default: chunk_sumsq_thread<GCLIP_BF16, M>(acc, c.addr, c.numel, s, st, pol); break;
  }
}

// The sum of squares of one chunk, valid in thread 0.
template <class M>
__device__ __forceinline__ SumSq chunk_sumsq(const clip_chunk_t& c, float s, float st, SumSq* red,
                                             uint64_t pol) {
  SumSq acc = {{0.f, 0.f}, {0.f, 0.f}};
  chunk_accumulate<M>(acc, c, s, st, pol);
  return block_reduce(acc, red);
}

__device__ __forceinline__ float4 pack(SumSq a) {
  return make_float4(a.big.hi, a.big.lo, a.tiny.hi, a.tiny.lo);
}

// ---------------------------------------------------------------------------
// The last microbatch's accumulation fused into the norm pass: every element
// of a chunk becomes x + a (a from the addend tensor at the same offset),
// rounded once to the format and stored back, and its square joins this
// thread's accumulator in the order chunk_sumsq_thread uses (vectors
// threadIdx.x, threadIdx.x + kThreads, ..., then the head element, then the
// tail element), so the norm equals that of a separate += followed by the
// clip.  An addend whose offset within 16 bytes differs from its gradient's
// is read element by element; the order of the arithmetic is the same.

constexpr int kAddUnroll = 2;  // vector pairs in flight per thread

// 16 bytes of elements from an address aligned only to the element size.
template <int DT>
__device__ __forceinline__ uint4 load_vec_elems(uint64_t a) {
  if constexpr (Fmt<DT>::kBytes == 4) {
    const unsigned int* p = reinterpret_cast<const unsigned int*>(a);
    return make_uint4(__ldcs(p), __ldcs(p + 1), __ldcs(p + 2), __ldcs(p + 3));
  } else {
    const unsigned short* p = reinterpret_cast<const unsigned short*>(a);
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      w[k] = static_cast<uint32_t>(__ldcs(p + 2 * k)) |
             (static_cast<uint32_t>(__ldcs(p + 2 * k + 1)) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// One scalar element: x + a rounded to the format, stored, squared.
template <int DT>
__device__ __forceinline__ void add_sumsq1(SumSq& acc, uint64_t x_at, uint64_t a_at, float s,
                                           float st) {
  const float r = Fmt<DT>::round1(__fadd_rn(Fmt<DT>::load1(x_at), Fmt<DT>::load1(a_at)));
  Fmt<DT>::store1(x_at, r);
  elem_sumsq(acc, r, s, st);
}

template <int DT>
__device__ __forceinline__ void chunk_add_sumsq_thread(SumSq& acc, uint64_t addr, uint64_t add_addr,
                                                       uint32_t n, float s, float st, uint64_t pol) {
  constexpr uint32_t B = Fmt<DT>::kBytes;
  const Span sp = make_span<DT>(addr, n);
  uint4* v = reinterpret_cast<uint4*>(sp.body);
  const uint64_t add_body = add_addr + static_cast<uint64_t>(sp.head) * B;
  const bool aligned = (add_body & 15u) == 0;  // the same in every thread
  const uint4* av = reinterpret_cast<const uint4*>(add_body);
  const uint64_t pol_add = policy_evict_first();  // the addend is read once
  for (uint32_t base = threadIdx.x; base < sp.nvec; base += kAddUnroll * kThreads) {
    uint4 x[kAddUnroll], a[kAddUnroll];
#pragma unroll
    for (int u = 0; u < kAddUnroll; ++u) {
      const uint32_t i = base + u * kThreads;
      x[u] = make_uint4(0, 0, 0, 0);
      a[u] = make_uint4(0, 0, 0, 0);
      if (i < sp.nvec) {
        x[u] = HintMem::ld(v + i, pol);
        a[u] = aligned ? HintMem::ld(av + i, pol_add)
                       : load_vec_elems<DT>(add_body + static_cast<uint64_t>(i) * 16u);
      }
    }
#pragma unroll
    for (int u = 0; u < kAddUnroll; ++u) {
      const uint32_t i = base + u * kThreads;
      if (i < sp.nvec) {
        const uint4 sum = Fmt<DT>::add(x[u], a[u]);
        HintMem::st_scale(v + i, sum, pol);
        vec_sumsq<DT>(acc, sum, s, st);
      }
    }
  }
  if (threadIdx.x < sp.head)
    add_sumsq1<DT>(acc, addr + threadIdx.x * B, add_addr + threadIdx.x * B, s, st);
  if (threadIdx.x < sp.ntail) {
    const uint64_t off = static_cast<uint64_t>(sp.tail_start + threadIdx.x) * B;
    add_sumsq1<DT>(acc, addr + off, add_addr + off, s, st);
  }
}

__device__ __forceinline__ void chunk_add_accumulate(SumSq& acc, const clip_chunk_t& c,
                                                     uint64_t add_addr, float s, float st,
                                                     uint64_t pol) {
  switch (c.meta & 0xffu) {
    case GCLIP_F32: chunk_add_sumsq_thread<GCLIP_F32>(acc, c.addr, add_addr, c.numel, s, st, pol); break;
    case GCLIP_F16: chunk_add_sumsq_thread<GCLIP_F16>(acc, c.addr, add_addr, c.numel, s, st, pol); break;
    default: chunk_add_sumsq_thread<GCLIP_BF16>(acc, c.addr, add_addr, c.numel, s, st, pol); break;
  }
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
// An entry is one SumSq packed as float4 {big.hi, big.lo, tiny.hi, tiny.lo}.
//
// The decision (decide_write) is taken in float-float arithmetic, or in
// double when the tiny bin is not empty, and the multiplier inv_scale *
// max_norm / norm is handed to the scaling pass as a float-float pair so
// that each output is rounded once.

__device__ SumSq reduce_partials(const float4* partials, int64_t n, SumSq* red) {
  SumSq acc = {{0.f, 0.f}, {0.f, 0.f}};
  // Up to four entries loaded at once, then added in increasing index order:
  // thread t's sum is always entries t, t + kThreads, t + 2 kThreads, ...
  for (int64_t c = threadIdx.x; c < n; c += 4 * kThreads) {
    float4 p[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = c + u * kThreads;
      p[u] = i < n ? __ldcg(partials + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (c + u * kThreads < n) acc = sumsq_add(acc, SumSq{{p[u].x, p[u].y}, {p[u].z, p[u].w}});
  }
  return block_reduce(acc, red);
}

// Float-float steps of the decision, after Dekker ("A floating-point
// technique for extending the available precision", 1971): products made
// exact with a fused multiply-add; a square root and a quotient each taken
// as the fp32 result plus one correction from the exactly computed
// remainder, good to about 2^-46.  GB300 runs fp64 at a small fraction of
// its fp32 rate, and one thread's dependent chain of double square root and
// division sat on the critical path of every clip.

__device__ __forceinline__ FF two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return FF{p, __fmaf_rn(a, b, -p)};
}

// sqrt(a) for a normalized float-float a > 0 whose high part is normal.
__device__ __forceinline__ FF ff_sqrt(FF a) {
  const float s = __fsqrt_rn(a.hi);
  const FF p = two_prod(s, s);
  // a - s^2: a.hi - p.hi is exact (the two are within a factor of two)
  const float r = __fadd_rn(__fsub_rn(__fsub_rn(a.hi, p.hi), p.lo), a.lo);
  return ff_renorm(s, __fdiv_rn(r, __fmul_rn(2.0f, s)));
}

// m / n for a float m and a normalized float-float n > 0.
__device__ __forceinline__ FF ff_div(float m, FF n) {
  const float q = __fdiv_rn(m, n.hi);
  // m - q * n.hi is exact for a correctly rounded q
  const float r = __fsub_rn(__fmaf_rn(-q, n.hi, m), __fmul_rn(q, n.lo));
  return ff_renorm(q, __fdiv_rn(r, n.hi));
}

__device__ __forceinline__ FF ff_mul(FF a, float b) {
  const FF p = two_prod(a.hi, b);
  return ff_renorm(p.hi, __fmaf_rn(a.lo, b, p.lo));
}

// The norm, flag, decision and multiplier from the two-bin sum of squares
// (thread 0).  `tiny_exp` is the K of the call (the tiny bin holds squares
// scaled by 2^2K).  When the tiny bin is empty (the usual case) the sum is
// the float-float big bin and everything is done in float-float: the norm
// is compared with max_norm exactly as a float-float value, reported
// rounded to fp32, and the multiplier inv_scale * max_norm / norm is handed
// on as a float-float pair.  Otherwise the bins are combined and the same
// steps taken in double.
__device__ void decide_write(SumSq acc, float max_norm, float inv_scale, int tiny_exp,
                             clip_result_t* res, float* out_norm, int32_t* out_flag,
                             unsigned int calls) {
  bool nonfinite;
  int decision;
  float norm_f, s_hi, s_lo, chi = 1.0f, clo = 0.0f;
  // Float-float unless the tiny bin holds something or the sum is within
  // 2^8 of fp32's range (where the square root rounds to 2^64 and its exact
  // square would overflow); those cases take the double path.
  if (acc.tiny.hi == 0.0f && acc.tiny.lo == 0.0f && !(acc.big.hi > 0x1p120f)) {
    s_hi = acc.big.hi;
    s_lo = acc.big.lo;
    nonfinite = !isfinite(s_hi) || !isfinite(s_lo);  // finite and below 2^120 here: S < FLT_MAX
    if (nonfinite) {
      decision = GCLIP_DECISION_SKIP;
      norm_f = __fsqrt_rn(s_hi);
    } else if (s_hi == 0.0f) {
      decision = GCLIP_DECISION_PASS;
      norm_f = 0.0f;
      chi = inv_scale;
    } else {
      // a non-zero big bin holds vectors whose sums are at least 2^-100
      const FF n = ff_sqrt(acc.big);
      norm_f = n.hi;
      if (n.hi > max_norm || (n.hi == max_norm && n.lo > 0.0f)) {
        decision = GCLIP_DECISION_CLIP;
        const FF k = ff_mul(ff_div(max_norm, n), inv_scale);
        chi = k.hi;
        clo = k.lo;
      } else {
        decision = GCLIP_DECISION_PASS;
        chi = inv_scale;
      }
    }
  } else {
    const double big = static_cast<double>(acc.big.hi) + static_cast<double>(acc.big.lo);
    const double tiny = static_cast<double>(acc.tiny.hi) + static_cast<double>(acc.tiny.lo);
    const double S = big + ldexp(tiny, -2 * tiny_exp);
    nonfinite = !isfinite(acc.big.hi) || !isfinite(acc.big.lo) || !isfinite(acc.tiny.hi) ||
                !isfinite(acc.tiny.lo) || S > static_cast<double>(FLT_MAX);
    const double norm = sqrt(S);
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
    norm_f = __double2float_rn(norm);
    s_hi = __double2float_rn(S);
    s_lo = __double2float_rn(S - static_cast<double>(s_hi));
  }
  res->norm = norm_f;
  res->nonfinite = nonfinite ? 1 : 0;
  res->decision = decision;
  res->coef_hi = chi;
  res->coef_lo = clo;
  res->sumsq_hi = s_hi;
  res->sumsq_lo = s_lo;
  res->calls = calls + 1u;  // `calls`: the count read before the reduction
  if (out_norm) *out_norm = norm_f;
  if (out_flag) *out_flag = nonfinite ? 1 : 0;
}

__device__ void final_reduce(const float4* partials, int64_t n, float max_norm, float inv_scale,
                             int tiny_exp, clip_result_t* res, float* out_norm, int32_t* out_flag,
                             SumSq* red) {
  // The record's call count, loaded now so that its latency overlaps the
  // reduction instead of following it.
  const unsigned int calls = threadIdx.x == 0 ? __ldcg(&res->calls) : 0u;
  const SumSq acc = reduce_partials(partials, n, red);
  if (threadIdx.x == 0)
    decide_write(acc, max_norm, inv_scale, tiny_exp, res, out_norm, out_flag, calls);
}

// ---------------------------------------------------------------------------
// Where a kernel finds chunk c: the handle's chunk table, or one contiguous
// buffer cut on the fly exactly as the host planner cuts a single tensor
// (the first chunk takes the elements before the first 16-byte boundary
// plus a full chunk, every later chunk starts aligned).

struct TableChunks {
  const clip_chunk_t* chunks;
  __device__ __forceinline__ clip_chunk_t operator[](int64_t c) const { return chunks[c]; }
};

struct FlatChunks {
  uint64_t base;
  int64_t numel;
  int32_t dtype;
  __device__ __forceinline__ clip_chunk_t operator[](int64_t c) const {
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
};

// ---------------------------------------------------------------------------
// The norm pass of the handle-based clip, shared by the register-engine
// variants (split, split_wave, single launch).
//
// Sets between half of L2 and four times L2 are also prefetched a chunk
// ahead into L2 (one bulk request per chunk, at normal priority, where the
// loads themselves ask for evict_first).  Measured on GB300: 120M fp32 clip
// -0.6 us, fp16 / bf16 sets -3 us, a skipped fp16 clip +0.7 us; most likely
// the prefetched lines of the last chunks are still in L2 when the scaling
// pass, which visits them first, starts.  On a 4.9 GB set the extra requests
// cost 1%, so larger sets are not prefetched.  The arithmetic is unchanged.
//
// A grid of G blocks (G fixed per handle).  Block b takes chunks b, b + G,
// b + 2G, ...; each of its threads keeps one two-bin accumulator over its
// share of all those chunks, in that order, and the block tree combines the
// threads once at the end.  The block sum goes to block_sums[b]; the block
// that arrives last reduces the G block sums in fixed order (final_reduce)
// and publishes the record.  Which block arrives last depends on timing; the
// arithmetic does not.

struct NormArgs {
  const clip_chunk_t* chunks;
  int64_t n_chunks;
  float4* block_sums;     // G entries
  unsigned int* arrive;   // blocks done with the norm pass in this call
  unsigned int* work;     // chunks the scaling pass claims in this call
  unsigned int expected;  // G, plus the test hook's extra arrivals
  float max_norm;
  float inv_scale;
  float inv_scale_tiny;   // inv_scale * 2^tiny_exp, exact
  int tiny_exp;
  clip_result_t* res;
  float* out_norm;
  int32_t* out_flag;
  int64_t keep_from;      // chunks from here on are read with evict_last
  int resident;           // the set fits in half of L2: the rest is read with evict_normal
  int prefetch;           // each block asks L2 for its next chunk ahead of its loads
  int32_t* hint;          // mapped host word: 1 if this clip writes, else 0 (may be NULL)
};

// One bulk request asking L2 for the aligned body of chunk `ch` (a hint: it
// reads nothing into registers).
__device__ __forceinline__ void prefetch_chunk_l2(const clip_chunk_t& ch) {
  const uint32_t es = (ch.meta & 0xffu) == GCLIP_F32 ? 4u : 2u;
  const uint32_t head = min(ch.numel, static_cast<uint32_t>(((16u - (ch.addr & 15u)) & 15u) / es));
  const uint32_t bytes = (ch.numel - head) / (16u / es) * 16u;
  if (bytes)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ch.addr + head * es), "r"(bytes)
                 : "memory");
}

// This block's chunk c: its share into `acc`, after a bulk L2 prefetch of
// the aligned body of its next chunk (when the set is prefetched).
__device__ __forceinline__ void norm_chunk(const NormArgs& a, int64_t c, const clip_chunk_t& ch,
                                           SumSq& acc, uint64_t pol_first, uint64_t pol_last) {
  if (a.prefetch && threadIdx.x == 0 && c + gridDim.x < a.n_chunks)
    prefetch_chunk_l2(a.chunks[c + gridDim.x]);
  chunk_accumulate<HintMem>(acc, ch, a.inv_scale, a.inv_scale_tiny,
                            c >= a.keep_from ? pol_last : pol_first);
}

__device__ __forceinline__ SumSq block_norm_pass(const NormArgs& a, SumSq* red) {
  // A set that fits in L2 may stay there for the next call; a larger one is
  // streamed through without displacing anything.
  const uint64_t pol_first = a.resident ? policy_evict_normal() : policy_evict_first();
  const uint64_t pol_last = policy_evict_last();
  SumSq acc = {{0.f, 0.f}, {0.f, 0.f}};
  for (int64_t c = blockIdx.x; c < a.n_chunks; c += gridDim.x)
    norm_chunk(a, c, a.chunks[c], acc, pol_first, pol_last);
  return block_reduce(acc, red);
}

// Publish this block's sum; returns true (in every thread) in the block that
// arrived last, after it has written the record.
__device__ __forceinline__ bool norm_arrive(const NormArgs& a, SumSq bsum, SumSq* red, int* s_flag) {
  if (threadIdx.x == 0) {
    a.block_sums[blockIdx.x] = pack(bsum);
    // One acquire-release ticket: the release publishes this block's sum
    // with the increment; the acquire in the block that takes the last
    // ticket makes every earlier block's sum visible to it (the increments
    // form one release sequence), and the barrier below passes that on to
    // the block's other threads.
    unsigned int t;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(t) : "l"(a.arrive) : "memory");
    *s_flag = (t + 1u == a.expected);
  }
  __syncthreads();
  if (!*s_flag) return false;
  final_reduce(a.block_sums, gridDim.x, a.max_norm, a.inv_scale, a.tiny_exp, a.res, a.out_norm,
               a.out_flag, red);
  if (threadIdx.x == 0) {
    // For the host's choice of the next call's scaling launch (this thread
    // wrote the record just now).
    if (a.hint != nullptr)
      *reinterpret_cast<volatile int32_t*>(a.hint) =
          must_write(a.res->decision, a.res->coef_hi, a.res->coef_lo) ? 1 : 0;
    // No fence: the end of the kernel orders these stores and the record
    // before the dependent launch; the single-launch kernels fence before
    // they release the other blocks.
    *a.arrive = 0u;  // every block has arrived: rearm for the next call
    *a.work = 0u;    // no scaling block claims before the record is out
  }
  return true;
}

}  // namespace gclip
