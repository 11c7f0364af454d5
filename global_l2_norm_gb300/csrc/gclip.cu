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
// This file keeps that pipeline as written (GCLIP_VARIANT_THREE_KERNEL), runs
// it by default in two launches (the last block of the partial-sum kernel
// does the final reduction), and adds a single-launch variant in which the
// last block to finish its partial sums reduces and releases the others to
// scale (the page's heading "Why three kernels and not one?" has no body, so
// the page gives no reason against it).
//
// The variants share every piece of arithmetic: the sums of squares (a fixed
// mapping of elements to the 256 threads of a block, fp32 squares into two
// float-float bins, a fixed shuffle tree) and the final reduction (a fixed
// strided order over the partial sums, the same tree, the decision), so the
// norm is bit-identical from run to run, and between the variants that cut
// the partial sums the same way.  The work is a streaming reduction bounded
// by HBM bandwidth; no tensor cores are used.
//
// Layout: common.cuh (float-float arithmetic, element formats, memory
// policies), reduce.cuh (chunk sums, block tree, final reduction, norm pass),
// kernels.cuh (register-engine kernels), tma.cuh (bulk-copy engine); this
// file holds the C ABI and the no-allocation entry point.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "internal.hpp"
#include "tma.cuh"


// ===========================================================================
// Host side: the C ABI.

using gclip::SyncWords;

struct gclip_handle {
  int device;
  int64_t n_chunks;
  int64_t total_bytes;       // bytes of all gradients
  int64_t keep_from;         // first chunk the norm pass reads with evict_last
  int64_t l2_bytes;          // L2 size of the device
  int32_t variant;
  int32_t grid_persistent;   // blocks of the register engine's norm pass (co-resident)
  int32_t grid_wave;         // blocks of a scaling wave (co-resident)
  int32_t grid_tma;          // blocks of the TMA engine (co-resident)
  int32_t coop;
  int32_t debug_extra;
  long long timeout_ns;
  void* arena;
  clip_chunk_t* d_chunks;
  float4* d_partials;        // one two-bin sum per chunk (per-chunk kernels) or per
                             // block of the norm pass (G <= chunks)
  clip_result_t* d_result;
  SyncWords* d_sync;
  clip_result_t* d_unit;     // a constant record: PASS, multiplier 1 (clip_adamw_step)
  int64_t* d_first;          // first chunk of each tensor, n_tensors + 1 entries
  clip_result_t* d_trec;     // per-tensor records of clip_grad_norm_per_tensor
  int64_t* d_wlist;          // chunks clip_grad_norm_per_tensor rewrites (n_chunks entries)
  unsigned int* d_wcount;    // length of that list, entries claimed from it
  std::vector<clip_tensor_desc_t> descs;   // the gradient tensors, as created
  gclip::TensorState* d_states;            // AdamW state table (NULL until attached)
  gclip::TensorState* d_outs;              // fp32 output table (NULL until attached)
  gclip::TensorState* d_adds;              // addend table (NULL until attached)
  // Pinned, mapped host word that the norm pass's last block sets to 1 when
  // the clip writes and to 0 when it does not; SPLIT reads it (without
  // waiting) to choose the shape of the next call's scaling launch.
  int32_t* h_hint;
  int32_t* d_hint;
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

// The tiny bin's multiplier inv_scale * 2^K and K: K = kTinyExpMax unless
// that product would exceed 2^126 (exact: a power-of-two scaling).
struct TinyScale {
  float st;
  int k;
};

TinyScale tiny_scale(float inv_scale) {
  int k = gclip::kTinyExpMax;
  double st = std::ldexp(static_cast<double>(inv_scale), k);
  while (k > 0 && st > 0x1p126) {
    --k;
    st *= 0.5;
  }
  return TinyScale{static_cast<float>(st), k};
}

// Blocks of a grid that strides over n chunks with at most `resident`
// blocks: the fewest that keep the largest share ceil(n / resident), so
// that every block gets the same number of chunks or one less.
int32_t balanced_grid(int64_t resident, int64_t n) {
  if (resident <= 0 || n <= 0) return static_cast<int32_t>(resident < n ? resident : n);
  const int64_t per = (n + resident - 1) / resident;
  return static_cast<int32_t>((n + per - 1) / per);
}

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
  a.work = &h->d_sync->work;
  a.expected = static_cast<unsigned int>(grid) + extra;
  a.max_norm = max_norm;
  a.inv_scale = inv_scale;
  const TinyScale ts = tiny_scale(inv_scale);
  a.inv_scale_tiny = ts.st;
  a.tiny_exp = ts.k;
  a.res = h->d_result;
  a.out_norm = out_norm;
  a.out_flag = out_flag;
  a.keep_from = h->keep_from;
  a.hint = h->d_hint;
  a.resident = h->total_bytes <= h->l2_bytes / 2 ? 1 : 0;
  a.prefetch = !a.resident && h->total_bytes <= 4 * h->l2_bytes ? 1 : 0;
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
  for (int32_t t = 0; t < n_tensors; ++t)
    h->total_bytes += descs[t].numel * (descs[t].dtype == GCLIP_F32 ? 4 : 2);
  h->variant = GCLIP_VARIANT_SPLIT;
  h->descs.assign(descs, descs + n_tensors);
  h->timeout_ns = gclip::kDefaultTimeoutNs;

  const size_t n = chunks.size();
  // G, the norm pass's grid, is known only after the occupancy query below;
  // it is at most the number of chunks, so size the block sums for that.
  const size_t off_chunks = 0;
  const size_t off_partials = round_up(off_chunks + n * sizeof(clip_chunk_t), 256);
  const size_t off_result = round_up(off_partials + n * sizeof(float4), 256);
  const size_t off_sync = round_up(off_result + sizeof(clip_result_t), 256);
  const size_t nt = static_cast<size_t>(n_tensors);
  const size_t off_first = round_up(off_sync + sizeof(SyncWords), 256);
  const size_t off_trec = round_up(off_first + (nt + 1) * sizeof(int64_t), 256);
  const size_t off_wlist = round_up(off_trec + (nt ? nt : 1) * sizeof(clip_result_t), 256);
  const size_t off_wcount = round_up(off_wlist + (n ? n : 1) * sizeof(int64_t), 256);
  const size_t off_unit = round_up(off_wcount + 2 * sizeof(unsigned int), 256);
  const size_t total = round_up(off_unit + sizeof(clip_result_t), 256);
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
  h->d_partials = reinterpret_cast<float4*>(base + off_partials);
  h->d_result = reinterpret_cast<clip_result_t*>(base + off_result);
  h->d_sync = reinterpret_cast<SyncWords*>(base + off_sync);
  h->d_first = reinterpret_cast<int64_t*>(base + off_first);
  h->d_trec = reinterpret_cast<clip_result_t*>(base + off_trec);
  h->d_wlist = reinterpret_cast<int64_t*>(base + off_wlist);
  h->d_wcount = reinterpret_cast<unsigned int*>(base + off_wcount);
  h->d_unit = reinterpret_cast<clip_result_t*>(base + off_unit);

  int sms = 0, per_sm = 0, coop = 0, l2 = 0;
  e = cudaMemset(h->arena, 0, total);
  if (e == cudaSuccess && n > 0)
    e = cudaMemcpy(h->d_chunks, chunks.data(), n * sizeof(clip_chunk_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(h->d_first, first.data(), first.size() * sizeof(int64_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) {
    clip_result_t unit = {};
    unit.decision = GCLIP_DECISION_PASS;
    unit.coef_hi = 1.0f;
    e = cudaMemcpy(h->d_unit, &unit, sizeof(unit), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, h->device);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gclip::k_clip_persistent,
                                                      gclip::kThreads, 0);
  int per_sm_tma = 0, per_sm_wave = 0;
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_wave, gclip::k_grad_scale_wave,
                                                      gclip::kThreads, 0);
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
  h->grid_persistent = balanced_grid(static_cast<int64_t>(sms) * per_sm, h->n_chunks);
  h->grid_tma = balanced_grid(static_cast<int64_t>(sms) * per_sm_tma, h->n_chunks);
  const int64_t wave = static_cast<int64_t>(sms) * per_sm_wave;
  h->grid_wave = static_cast<int32_t>(wave < h->n_chunks ? wave : h->n_chunks);
  h->coop = coop;
  // The write hint: without it SPLIT always scales with one block per chunk.
  if (cudaHostAlloc(reinterpret_cast<void**>(&h->h_hint), 64, cudaHostAllocMapped) == cudaSuccess) {
    *h->h_hint = 1;
    if (cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->d_hint), h->h_hint, 0) != cudaSuccess) {
      cudaFreeHost(h->h_hint);
      h->h_hint = h->d_hint = nullptr;
    }
  }
  cudaGetLastError();
  *out = h;
  return GCLIP_OK;
}

namespace {

// The in-place scaling pass of the split variants, after the norm pass:
// one block per chunk, or one resident wave that claims chunks.  SPLIT_WAVE
// always takes the wave.  SPLIT takes the wave when the last norm pass that
// has completed on this handle decided to write nothing (the hint word, read
// without synchronising; the calls enqueued since may not have run yet):
// when nothing is written, the wave retires ~760 blocks instead of one per
// chunk, and when everything is, one block per chunk is 1.5% faster.  Both
// kernels give the same results bit for bit, so a wrong guess costs time
// only.
//
// `after_norm_pass`: the norm pass was k_grad_norm_partial, so one block per
// chunk may be k_grad_scale_early, whose first wave loads its chunks before
// the decision is out (measured on GB300, ANDREA-120M: a writing clip 161.0
// -> 159.7 us, fp16 81.9 -> 81.0, tiny 7.4 -> 6.7; a no-write clip after a
// writing one costs the same as before).
cudaError_t launch_scale(clip_handle_t h, cudaStream_t s, bool pdl, bool after_norm_pass = false) {
  const clip_chunk_t* chunks = h->d_chunks;
  int64_t nc = h->n_chunks;
  const clip_result_t* cres = h->d_result;
  const bool wave = h->variant == GCLIP_VARIANT_SPLIT_WAVE ||
                    (h->variant == GCLIP_VARIANT_SPLIT && h->h_hint != nullptr &&
                     *reinterpret_cast<volatile int32_t*>(h->h_hint) == 0);
  if (wave) {
    unsigned int* work = &h->d_sync->work;
    void* args[] = {&chunks, &nc, &cres, &work};
    return launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_scale_wave),
                      static_cast<unsigned int>(h->grid_wave), s, args, pdl);
  }
  if (after_norm_pass) {
    // the first resident wave of one-chunk scaling blocks
    unsigned int n_early = static_cast<unsigned int>(h->grid_wave);
    void* args[] = {&chunks, &nc, &cres, &n_early};
    return launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_scale_early),
                      static_cast<unsigned int>(nc), s, args, pdl);
  }
  gclip::TableChunks src{chunks};
  void* args[] = {&src, &nc, &cres};
  return launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_scale<gclip::TableChunks>),
                    static_cast<unsigned int>(nc), s, args, pdl);
}

// The final reduction alone, for a set with no chunks (norm 0, PASS).
cudaError_t launch_empty(clip_handle_t h, float max_norm, float inv_scale, float* out_norm,
                         int32_t* out_flag, cudaStream_t s) {
  const float4* partials = h->d_partials;
  int64_t n = 0;
  int k = tiny_scale(inv_scale).k;
  void* args[] = {&partials, &n, &max_norm, &inv_scale, &k, &h->d_result, &out_norm, &out_flag};
  return launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_final), 1, s, args, false);
}

// Enqueue one clip.  `events` (may be NULL) are recorded between the steps;
// programmatic dependent launch is used only when no events are recorded.
int enqueue(clip_handle_t h, float max_norm, float inv_scale, float* out_norm,
            int32_t* out_flag, cudaStream_t s, cudaEvent_t const* events) {
  int64_t nc = h->n_chunks;
  const float4* partials = h->d_partials;
  const bool pdl = events == nullptr;
  cudaError_t e = cudaSuccess;
  auto mark = [&](int i) {
    if (events != nullptr && e == cudaSuccess) e = cudaEventRecord(events[i], s);
  };

  mark(0);
  if (nc == 0) {
    mark(1);
    mark(2);
    if (e == cudaSuccess) e = launch_empty(h, max_norm, inv_scale, out_norm, out_flag, s);
  } else if (h->variant == GCLIP_VARIANT_THREE_KERNEL) {
    // The clipping page's pipeline as written: per-chunk sums, one block that
    // reduces them and decides, one block per chunk that scales.
    const TinyScale ts = tiny_scale(inv_scale);
    gclip::TableChunks src{h->d_chunks};
    float4* parts = h->d_partials;
    unsigned int* no_clear = nullptr;
    int resident = h->total_bytes <= h->l2_bytes / 2 ? 1 : 0;
    float st = ts.st;
    int k = ts.k;
    void* a1[] = {&src, &inv_scale, &st, &parts, &no_clear, &resident};
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_chunk_sums<gclip::TableChunks>),
                     static_cast<unsigned int>(nc), s, a1, pdl);
    mark(1);
    void* a2[] = {&partials, &nc, &max_norm, &inv_scale, &k, &h->d_result, &out_norm, &out_flag};
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_final), 1, s, a2, pdl);
    mark(2);
    if (e == cudaSuccess) e = launch_scale(h, s, pdl);
  } else if (h->variant == GCLIP_VARIANT_SPLIT || h->variant == GCLIP_VARIANT_SPLIT_WAVE) {
    gclip::NormArgs a = norm_args(h, h->grid_persistent, max_norm, inv_scale, out_norm, out_flag, 0);
    void* a1[] = {&a};
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_partial),
                     static_cast<unsigned int>(h->grid_persistent), s, a1, pdl);
    mark(1);
    mark(2);
    if (e == cudaSuccess) e = launch_scale(h, s, pdl, true);
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
    if (h->d_adds != nullptr && cudaFree(h->d_adds) != cudaSuccess) rc = GCLIP_ERR_CUDA;
    if (h->h_hint != nullptr && cudaFreeHost(h->h_hint) != cudaSuccess) rc = GCLIP_ERR_CUDA;
    cudaGetLastError();
  }
  delete h;
  return rc;
}

extern "C" int clip_set_variant(clip_handle_t h, int32_t variant) {
  if (h == nullptr) return GCLIP_ERR_INVALID_ARG;
  if (variant < GCLIP_VARIANT_SPLIT || variant > GCLIP_VARIANT_THREE_KERNEL)
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

extern "C" int clip_last_status(clip_handle_t h, int32_t* d_out, void* stream) {
  if (h == nullptr || d_out == nullptr) return GCLIP_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok) return GCLIP_ERR_CUDA;
  const cudaError_t e = cudaMemcpyAsync(d_out, &h->d_result->status, sizeof(int32_t),
                                        cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream));
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

// Validate per-tensor arrays (`per` of them for each tensor, `ptrs` laid out
// tensor by tensor; fp32, or of the gradient's own format with grad_dtype)
// against the handle's gradients, and replace *slot with a device table of
// {gradient base, arrays...}.
int attach_table(clip_handle_t h, const void* const* ptrs, int per, int32_t n_tensors,
                 gclip::TensorState** slot, bool grad_dtype = false) {
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
      const void* a = ptrs[static_cast<size_t>(t) * per + k];
      f[k] = reinterpret_cast<uint64_t>(a);
      if (d.numel == 0) continue;
      clip_tensor_desc_t s = {const_cast<void*>(a), d.numel, grad_dtype ? d.dtype : GCLIP_F32, 0};
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
    e = launch_empty(h, max_norm, inv_scale, out_norm, out_flag, s);
  } else {
    gclip::NormArgs a = norm_args(h, h->grid_persistent, max_norm, inv_scale, out_norm, out_flag, 0);
    void* a1[] = {&a};
    e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_partial),
                   static_cast<unsigned int>(h->grid_persistent), s, a1, true);
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
  return attach_table(h, reinterpret_cast<const void* const*>(ptrs.data()), 3, n_tensors,
                      &h->d_states);
}

extern "C" int clip_attach_f32_out(clip_handle_t h, float* const* outs, int32_t n_tensors) {
  if (h == nullptr) return GCLIP_ERR_INVALID_ARG;
  return attach_table(h, const_cast<const void* const*>(reinterpret_cast<void* const*>(outs)), 1,
                      n_tensors, &h->d_outs);
}

extern "C" int clip_attach_addend(clip_handle_t h, const void* const* addends, int32_t n_tensors) {
  if (h == nullptr) return GCLIP_ERR_INVALID_ARG;
  return attach_table(h, addends, 1, n_tensors, &h->d_adds, true);
}

extern "C" int clip_grad_norm_accumulate(clip_handle_t h, float max_norm, float inv_scale,
                                         float* out_norm, int32_t* out_nonfinite_flag,
                                         void* stream) {
  if (h == nullptr || h->d_adds == nullptr || !valid_scalar(max_norm) || !valid_scalar(inv_scale))
    return GCLIP_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok) return GCLIP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int64_t nc = h->n_chunks;
  cudaError_t e = cudaSuccess;
  if (nc == 0) {
    e = launch_empty(h, max_norm, inv_scale, out_norm, out_nonfinite_flag, s);
  } else {
    gclip::NormArgs a =
        norm_args(h, h->grid_persistent, max_norm, inv_scale, out_norm, out_nonfinite_flag, 0);
    const gclip::TensorState* adds = h->d_adds;
    void* a1[] = {&a, &adds};
    e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_accumulate),
                   static_cast<unsigned int>(h->grid_persistent), s, a1, true);
    if (e == cudaSuccess) e = launch_scale(h, s, true);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GCLIP_ERR_CUDA;
  }
  return GCLIP_OK;
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

namespace {

// The AdamW hyperparameters of step `step` as the kernel takes them; false
// if one is out of range.
bool adamw_args(const clip_adamw_params_t* p, int64_t step, gclip::AdamwArgs& q) {
  const bool ok = step >= 1 && std::isfinite(p->lr) && p->lr >= 0.0f && std::isfinite(p->eps) &&
                  p->eps > 0.0f && std::isfinite(p->weight_decay) && p->weight_decay >= 0.0f &&
                  p->beta1 >= 0.0f && p->beta1 < 1.0f && p->beta2 >= 0.0f && p->beta2 < 1.0f;
  if (!ok) return false;
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
  return true;
}

}  // namespace

extern "C" int clip_grad_norm_adamw(clip_handle_t h, float max_norm, float inv_scale,
                                    const clip_adamw_params_t* p, int64_t step, float* out_norm,
                                    int32_t* out_nonfinite_flag, void* stream) {
  if (h == nullptr || p == nullptr || h->d_states == nullptr || !valid_scalar(max_norm) ||
      !valid_scalar(inv_scale))
    return GCLIP_ERR_INVALID_ARG;
  gclip::AdamwArgs q;
  if (!adamw_args(p, step, q)) return GCLIP_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok) return GCLIP_ERR_CUDA;
  int64_t nc = h->n_chunks;
  const clip_chunk_t* chunks = h->d_chunks;
  const gclip::TensorState* st = h->d_states;
  const clip_result_t* cres = h->d_result;
  void* args[] = {&chunks, &nc, &st, &cres, &q};
  return enqueue_norm_then(h, max_norm, inv_scale, out_norm, out_nonfinite_flag,
                           static_cast<cudaStream_t>(stream),
                           reinterpret_cast<const void*>(gclip::k_adamw), args);
}

extern "C" int clip_adamw_step(clip_handle_t h, const clip_adamw_params_t* p, int64_t step,
                               void* stream) {
  if (h == nullptr || p == nullptr || h->d_states == nullptr) return GCLIP_ERR_INVALID_ARG;
  gclip::AdamwArgs q;
  if (!adamw_args(p, step, q)) return GCLIP_ERR_INVALID_ARG;
  int64_t nc = h->n_chunks;
  if (nc == 0) return GCLIP_OK;
  DeviceGuard guard(h->device);
  if (!guard.ok) return GCLIP_ERR_CUDA;
  const clip_chunk_t* chunks = h->d_chunks;
  const gclip::TensorState* st = h->d_states;
  const clip_result_t* unit = h->d_unit;
  void* args[] = {&chunks, &nc, &st, &unit, &q};
  if (launch_pdl(reinterpret_cast<const void*>(gclip::k_adamw), static_cast<unsigned int>(nc),
                 static_cast<cudaStream_t>(stream), args, true) != cudaSuccess) {
    cudaGetLastError();
    return GCLIP_ERR_CUDA;
  }
  return GCLIP_OK;
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
  float4* partials = h->d_partials;
  const float4* cpartials = partials;
  const int64_t* first = h->d_first;
  clip_result_t* recs = h->d_trec;
  const clip_result_t* crecs = recs;
  int64_t* wlist = h->d_wlist;
  const int64_t* cwlist = wlist;
  unsigned int* wcount = h->d_wcount;
  cudaError_t e = cudaSuccess;
  const TinyScale ts = tiny_scale(inv_scale);
  float st = ts.st;
  int k = ts.k;
  if (nc > 0) {
    // Not a programmatic dependent: it empties the write list, which the
    // previous call's scaling kernel reads until it ends.
    gclip::TableChunks src{chunks};
    int resident = 0;
    void* a1[] = {&src, &inv_scale, &st, &partials, &wcount, &resident};
    e = launch_pdl(reinterpret_cast<const void*>(gclip::k_chunk_sums<gclip::TableChunks>),
                   static_cast<unsigned int>(nc), s, a1, false);
  }
  void* a2[] = {&cpartials, &first, &max_norm, &inv_scale, &k, &recs,
                &out_norms, &out_nonfinite_flags, &wlist, &wcount};
  if (e == cudaSuccess)
    e = launch_pdl(reinterpret_cast<const void*>(gclip::k_tensor_final), nt, s, a2, nc > 0);
  void* a3[] = {&chunks, &cwlist, &wcount, &crecs};
  if (e == cudaSuccess && nc > 0)
    e = launch_pdl(reinterpret_cast<const void*>(gclip::k_scale_per_tensor),
                   static_cast<unsigned int>(h->grid_wave), s, a3, true);
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

// The scratch of clip_grad_norm_flat_noalloc: one two-bin partial sum per
// chunk, then the result record.  Compiled into the library, so it costs
// every GPU that loads the library GCLIP_NOALLOC_SCRATCH_BYTES until exit.
constexpr size_t kNoAllocPartialBytes = static_cast<size_t>(GCLIP_NOALLOC_MAX_CHUNKS) * sizeof(float4);
static_assert(kNoAllocPartialBytes + sizeof(clip_result_t) <= GCLIP_NOALLOC_SCRATCH_BYTES,
              "record does not fit the scratch");
static __device__ __align__(256) unsigned char g_noalloc_scratch[GCLIP_NOALLOC_SCRATCH_BYTES];

}  // namespace gclip

namespace {

constexpr int kNoAllocMaxDevices = 64;

// What the entry point needs to know about a device, looked up once.
struct NoAllocDevice {
  char* scratch;  // device address of gclip::g_noalloc_scratch on that device
  int64_t l2;     // L2 size in bytes
};

std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc[kNoAllocMaxDevices];

// The set-up of device `dev` (the current device): the scratch array's
// device address and the L2 size, looked up on the first call and kept.
bool noalloc_device(int dev, NoAllocDevice* out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc[dev];
  if (d.scratch == nullptr) {
    void* p = nullptr;
    int l2 = 0;
    if (cudaGetSymbolAddress(&p, gclip::g_noalloc_scratch) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return false;
    }
    d.l2 = l2;
    d.scratch = static_cast<char*>(p);
  }
  *out = d;
  return true;
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
  NoAllocDevice d;
  if (!noalloc_device(dev, &d)) return GCLIP_ERR_CUDA;
  float4* partials = reinterpret_cast<float4*>(d.scratch);
  clip_result_t* record = reinterpret_cast<clip_result_t*>(d.scratch + gclip::kNoAllocPartialBytes);
  const float4* cpartials = partials;
  const TinyScale ts = tiny_scale(inv_scale);
  float st = ts.st;
  int k = ts.k;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;

  // The three launches of GCLIP_VARIANT_THREE_KERNEL, over chunks computed
  // from the buffer instead of read from a table.
  void* a2[] = {&cpartials, &nc, &max_norm, &inv_scale, &k, &record, &out_norm, &out_nonfinite_flag};
  if (nc == 0) {
    e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_final), 1, s, a2, false);
  } else {
    gclip::FlatChunks src{base, numel, dtype};
    unsigned int* no_clear = nullptr;
    int resident = numel * es <= d.l2 / 2 ? 1 : 0;
    void* a1[] = {&src, &inv_scale, &st, &partials, &no_clear, &resident};
    e = launch_pdl(reinterpret_cast<const void*>(gclip::k_chunk_sums<gclip::FlatChunks>),
                   static_cast<unsigned int>(nc), s, a1, false);
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_norm_final), 1, s, a2, true);
    const clip_result_t* crecord = record;
    void* a3[] = {&src, &nc, &crecord};
    if (e == cudaSuccess)
      e = launch_pdl(reinterpret_cast<const void*>(gclip::k_grad_scale<gclip::FlatChunks>),
                     static_cast<unsigned int>(nc), s, a3, true);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GCLIP_ERR_CUDA;
  }
  return GCLIP_OK;
}
