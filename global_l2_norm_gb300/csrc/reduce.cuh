// reduce.cuh -- the arithmetic of the norm: per-thread sums of squares of a
// chunk (plain, or with the last microbatch added in), the fixed block tree,
// the scaling of a chunk, the final reduction with the decision in double,
// and the norm pass shared by the register-engine variants.
// Included by gclip.cu only.
#pragma once

#include <cfloat>

#include "common.cuh"

namespace gclip {

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
__device__ __forceinline__ FF add_sumsq1(FF acc, uint64_t x_at, uint64_t a_at, float s) {
  const float r = Fmt<DT>::round1(__fadd_rn(Fmt<DT>::load1(x_at), Fmt<DT>::load1(a_at)));
  Fmt<DT>::store1(x_at, r);
  const float y = __fmul_rn(r, s);
  return ff_add_f(acc, __fmul_rn(y, y));
}

template <int DT>
__device__ __forceinline__ FF chunk_add_sumsq_thread(FF acc, uint64_t addr, uint64_t add_addr,
                                                     uint32_t n, float s, uint64_t pol) {
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
        acc = ff_add_f(acc, Fmt<DT>::sumsq(sum, s));
      }
    }
  }
  if (threadIdx.x < sp.head)
    acc = add_sumsq1<DT>(acc, addr + threadIdx.x * B, add_addr + threadIdx.x * B, s);
  if (threadIdx.x < sp.ntail) {
    const uint64_t off = static_cast<uint64_t>(sp.tail_start + threadIdx.x) * B;
    acc = add_sumsq1<DT>(acc, addr + off, add_addr + off, s);
  }
  return acc;
}

__device__ __forceinline__ FF chunk_add_accumulate(FF acc, const clip_chunk_t& c, uint64_t add_addr,
                                                   float s, uint64_t pol) {
  switch (c.meta & 0xffu) {
    case GCLIP_F32: return chunk_add_sumsq_thread<GCLIP_F32>(acc, c.addr, add_addr, c.numel, s, pol);
    case GCLIP_F16: return chunk_add_sumsq_thread<GCLIP_F16>(acc, c.addr, add_addr, c.numel, s, pol);
    default: return chunk_add_sumsq_thread<GCLIP_BF16>(acc, c.addr, add_addr, c.numel, s, pol);
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
//
// The decision is taken in double from the float-float sum: S = hi + lo is
// exact in double, norm = sqrt(S) and max_norm / norm are IEEE double
// operations, and the multiplier inv_scale * max_norm / norm is handed to the
// scaling pass as a float-float pair so that each output is rounded once.

__device__ FF reduce_partials(const float2* partials, int64_t n, FF* red) {
  FF acc = {0.f, 0.f};
  // Up to four entries loaded at once, then added in increasing index order:
  // thread t's sum is always entries t, t + kThreads, t + 2 kThreads, ...
  for (int64_t c = threadIdx.x; c < n; c += 4 * kThreads) {
    float2 p[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = c + u * kThreads;
      p[u] = i < n ? __ldcg(partials + i) : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (c + u * kThreads < n) acc = ff_add(acc, FF{p[u].x, p[u].y});
  }
  return block_reduce(acc, red);
}

// The norm, flag, decision and multiplier from the float-float sum of
// squares S = hi + lo (thread 0).
__device__ void decide_write(FF acc, float max_norm, float inv_scale, clip_result_t* res,
                             float* out_norm, int32_t* out_flag, unsigned int calls) {
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
  res->calls = calls + 1u;  // `calls`: the count read before the reduction
  if (out_norm) *out_norm = norm_f;
  if (out_flag) *out_flag = nonfinite ? 1 : 0;
}

__device__ void final_reduce(const float2* partials, int64_t n_chunks, float max_norm,
                             float inv_scale, clip_result_t* res, float* out_norm,
                             int32_t* out_flag, FF* red) {
  // The record's call count, loaded now so that its latency overlaps the
  // reduction instead of following it.
  const unsigned int calls = threadIdx.x == 0 ? __ldcg(&res->calls) : 0u;
  const FF acc = reduce_partials(partials, n_chunks, red);
  if (threadIdx.x == 0) decide_write(acc, max_norm, inv_scale, res, out_norm, out_flag, calls);
}

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
  unsigned int* work;     // chunks the scaling pass claims in this call
  unsigned int expected;  // G, plus the test hook's extra arrivals
  float max_norm;
  float inv_scale;
  clip_result_t* res;
  float* out_norm;
  int32_t* out_flag;
  int64_t keep_from;      // chunks from here on are read with evict_last
  int resident;           // the set fits in half of L2: the rest is read with evict_normal
  int prefetch;           // each block asks L2 for its next chunk ahead of its loads
};

__device__ __forceinline__ FF block_norm_pass(const NormArgs& a, FF* red) {
  // A set that fits in L2 may stay there for the next call; a larger one is
  // streamed through without displacing anything.
  const uint64_t pol_first = a.resident ? policy_evict_normal() : policy_evict_first();
  const uint64_t pol_last = policy_evict_last();
  FF acc = {0.f, 0.f};
  for (int64_t c = blockIdx.x; c < a.n_chunks; c += gridDim.x) {
    const clip_chunk_t ch = a.chunks[c];
    if (a.prefetch && threadIdx.x == 0 && c + gridDim.x < a.n_chunks) {
      // One bulk request for the aligned body of this block's next chunk.
      const clip_chunk_t nx = a.chunks[c + gridDim.x];
      const uint32_t es = (nx.meta & 0xffu) == GCLIP_F32 ? 4u : 2u;
      const uint32_t head = min(nx.numel, static_cast<uint32_t>(((16u - (nx.addr & 15u)) & 15u) / es));
      const uint32_t bytes = (nx.numel - head) / (16u / es) * 16u;
      if (bytes)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(nx.addr + head * es), "r"(bytes)
                     : "memory");
    }
    acc = chunk_accumulate<HintMem>(acc, ch, a.inv_scale, c >= a.keep_from ? pol_last : pol_first);
  }
  return block_reduce(acc, red);
}

// Publish this block's sum; returns true (in every thread) in the block that
// arrived last, after it has written the record.
__device__ __forceinline__ bool norm_arrive(const NormArgs& a, FF bsum, FF* red, int* s_flag) {
  if (threadIdx.x == 0) {
    a.block_sums[blockIdx.x] = make_float2(bsum.hi, bsum.lo);
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
  final_reduce(a.block_sums, gridDim.x, a.max_norm, a.inv_scale, a.res, a.out_norm, a.out_flag,
               red);
  if (threadIdx.x == 0) {
    // No fence: the end of the kernel orders these stores and the record
    // before the dependent launch; the single-launch kernels fence before
    // they release the other blocks.
    *a.arrive = 0u;  // every block has arrived: rearm for the next call
    *a.work = 0u;    // no scaling block claims before the record is out
  }
  return true;
}

}  // namespace gclip
