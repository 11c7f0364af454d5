// tma.cuh -- the TMA engine: the norm and scaling passes staged through
// shared memory by bulk copies (cp.async.bulk, mbarrier completion).
// Included by gclip.cu only.
#pragma once

#include "kernels.cuh"

namespace gclip {

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
// accumulators (vector j of the thread's share goes to big[j % 4]) so that
// four float-float chains run side by side; head and tail scalars go to
// big[0].  Vectors and scalars of tiny elements go to the one `tiny` bin
// (see SumSq).  The order is fixed, so the result is deterministic.
template <int DT>
__device__ __forceinline__ void stage_sumsq(FF (&big)[4], FF& tiny, const uint8_t* st,
                                            const clip_chunk_t& c, float s, float sti) {
  const Span sp = make_span<DT>(c.addr, c.numel);
  const uint4* v = reinterpret_cast<const uint4*>(st);
  uint32_t i = threadIdx.x;
  for (; i + 3 * kThreads < sp.nvec; i += 4 * kThreads) {
    const uint4 v0 = v[i], v1 = v[i + kThreads], v2 = v[i + 2 * kThreads], v3 = v[i + 3 * kThreads];
    vec_sumsq<DT>(big[0], tiny, v0, s, sti);
    vec_sumsq<DT>(big[1], tiny, v1, s, sti);
    vec_sumsq<DT>(big[2], tiny, v2, s, sti);
    vec_sumsq<DT>(big[3], tiny, v3, s, sti);
  }
  // fewer than four vectors left: constant indices keep the bins in registers
  if (i < sp.nvec) vec_sumsq<DT>(big[0], tiny, v[i], s, sti);
  if (i + kThreads < sp.nvec) vec_sumsq<DT>(big[1], tiny, v[i + kThreads], s, sti);
  if (i + 2 * kThreads < sp.nvec) vec_sumsq<DT>(big[2], tiny, v[i + 2 * kThreads], s, sti);
  constexpr uint32_t B = Fmt<DT>::kBytes;
  if (threadIdx.x < sp.head) elem_sumsq(big[0], tiny, Fmt<DT>::load1(c.addr + threadIdx.x * B), s, sti);
  if (threadIdx.x < sp.ntail)
    elem_sumsq(big[0], tiny,
               Fmt<DT>::load1(c.addr + static_cast<uint64_t>(sp.tail_start + threadIdx.x) * B), s, sti);
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
__device__ bool tma_norm_pass(const NormArgs& a, const Ring& r, uint32_t& phase, SumSq* red,
                              volatile int* s_abort, SumSq* out) {
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
  FF tiny = {0.f, 0.f};
  for (int64_t k = 0; k < mine; ++k) {
    const int s = static_cast<int>(k % kStages);
    if (ring_wait(r, k, phase, a.res, s_abort)) {
      const clip_chunk_t ch = a.chunks[norm_chunk(k)];
      switch (ch.meta & 0xffu) {
        case GCLIP_F32: stage_sumsq<GCLIP_F32>(acc, tiny, r.stage(s), ch, a.inv_scale, a.inv_scale_tiny); break;
        case GCLIP_F16: stage_sumsq<GCLIP_F16>(acc, tiny, r.stage(s), ch, a.inv_scale, a.inv_scale_tiny); break;
        default: stage_sumsq<GCLIP_BF16>(acc, tiny, r.stage(s), ch, a.inv_scale, a.inv_scale_tiny); break;
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
  *out = block_reduce(SumSq{ff_add(ff_add(acc[0], acc[1]), ff_add(acc[2], acc[3])), tiny}, red);
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
  __shared__ SumSq red[kWarps];
  __shared__ int s_abort, s_flag;
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) s_abort = 0;
  const Ring r = ring_setup(smem);
  uint32_t phase = 0;
  SumSq bsum;
  // A block whose copy timed out still arrives, with a NaN sum, so that the
  // record is published and says SKIP.
  if (!tma_norm_pass(a, r, phase, red, &s_abort, &bsum) && threadIdx.x == 0)
    bsum = SumSq{{__int_as_float(0x7fc00000), 0.f}, {0.f, 0.f}};
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
  __shared__ SumSq red[kWarps];
  __shared__ unsigned int s_gen0;
  __shared__ int s_abort, s_flag, s_go;
  if (threadIdx.x == 0) {
    s_gen0 = *reinterpret_cast<volatile unsigned int*>(&sync->gen);
    s_abort = 0;
  }
  const Ring r = ring_setup(smem);
  uint32_t phase = 0;
  SumSq bsum;
  const bool ok = tma_norm_pass(a, r, phase, red, &s_abort, &bsum);
  // A block whose copy timed out still arrives, with a NaN sum (so the clip
  // is skipped), to keep the others from waiting for it.
  if (!ok && threadIdx.x == 0) bsum = SumSq{{__int_as_float(0x7fc00000), 0.f}, {0.f, 0.f}};
  const bool published = norm_arrive(a, bsum, red, &s_flag);

  // Speculative prefetch of the scaling pass while the record is pending.
  int64_t issued = 0;
  if (threadIdx.x == 0 && ok) issued = tma_scale_prefetch(a.chunks, a.n_chunks, r, policy_evict_first());

  if (published) {
    if (threadIdx.x == 0) {
      __threadfence();  // the record before the generation that releases the others
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
