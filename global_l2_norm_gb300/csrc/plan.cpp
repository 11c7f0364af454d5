// plan.cpp -- host-side argument checks and the multi-tensor chunk table.
//
// The clipping page ("Grow a language model: gradient clipping",
// unhomeschool.com), section "ANDREA's three-kernel pipeline", cuts the work
// into fragments handled by one thread block each, hundreds of blocks over
// all tensors; section "Why computing the grad norm needs three kernels"
// names the obstacle this solves: tensors of very different shapes
// (embedding 8449x768, attention 768x768, layer norm 768) in one pass.  Here
// every tensor is cut into chunks of at most GCLIP_CHUNK_BYTES, in tensor
// order, so one launch covers the whole set and every block does about the
// same amount of work.  The table is built once (the backprop page, section
// "Cost of general frameworks": allocate everything at start-up).
#include "internal.hpp"

#include <algorithm>
#include <cstring>

namespace gclip {

int elem_size(int32_t dtype) {
  switch (dtype) {
    case GCLIP_F32: return 4;
    case GCLIP_F16:
    case GCLIP_BF16: return 2;
    default: return 0;
  }
}

int validate_descs(const clip_tensor_desc_t* descs, int32_t n) {
  if (n < 0 || n > GCLIP_MAX_TENSORS) return GCLIP_ERR_INVALID_ARG;
  if (n > 0 && descs == nullptr) return GCLIP_ERR_INVALID_ARG;
  struct Range { uint64_t lo, hi; };
  std::vector<Range> ranges;
  ranges.reserve(static_cast<size_t>(n));
  for (int32_t t = 0; t < n; ++t) {
    const clip_tensor_desc_t& d = descs[t];
    const int es = elem_size(d.dtype);
    if (es == 0 || d.numel < 0 || d.reserved != 0) return GCLIP_ERR_INVALID_ARG;
    if (d.numel == 0) continue;
    const uint64_t p = reinterpret_cast<uint64_t>(d.ptr);
    if (p == 0 || p % static_cast<uint64_t>(es) != 0) return GCLIP_ERR_INVALID_ARG;
    const uint64_t bytes = static_cast<uint64_t>(d.numel) * static_cast<uint64_t>(es);
    if (bytes / static_cast<uint64_t>(es) != static_cast<uint64_t>(d.numel) ||
        p + bytes < p)
      return GCLIP_ERR_INVALID_ARG;  // wraps the address space
    ranges.push_back({p, p + bytes});
  }
  std::sort(ranges.begin(), ranges.end(),
            [](const Range& a, const Range& b) { return a.lo < b.lo; });
  for (size_t i = 1; i < ranges.size(); ++i)
    if (ranges[i].lo < ranges[i - 1].hi) return GCLIP_ERR_INVALID_ARG;
  return GCLIP_OK;
}

int build_chunks(const clip_tensor_desc_t* descs, int32_t n,
                 std::vector<clip_chunk_t>& out) {
  const int rc = validate_descs(descs, n);
  if (rc != GCLIP_OK) return rc;
  out.clear();
  for (int32_t t = 0; t < n; ++t) {
    const clip_tensor_desc_t& d = descs[t];
    if (d.numel == 0) continue;
    const uint64_t es = static_cast<uint64_t>(elem_size(d.dtype));
    const uint64_t per_chunk = GCLIP_CHUNK_BYTES / es;
    const uint64_t base = reinterpret_cast<uint64_t>(d.ptr);
    const uint32_t meta = static_cast<uint32_t>(d.dtype) |
                          (static_cast<uint32_t>(t) << 8);
    // The first chunk also takes the elements before the first 16-byte
    // boundary, so that every later chunk starts aligned for vector loads.
    const uint64_t head = ((16 - base % 16) % 16) / es;
    uint64_t done = 0;
    const uint64_t total = static_cast<uint64_t>(d.numel);
    while (done < total) {
      const uint64_t want = (done == 0) ? head + per_chunk : per_chunk;
      const uint64_t m = std::min(want, total - done);
      clip_chunk_t c;
      c.addr = base + done * es;
      c.numel = static_cast<uint32_t>(m);
      c.meta = meta;
      out.push_back(c);
      done += m;
    }
  }
  return GCLIP_OK;
}

}  // namespace gclip

extern "C" int clip_plan(const clip_tensor_desc_t* descs, int32_t n_tensors,
                         clip_chunk_t* out, int64_t capacity, int64_t* n_chunks) {
  if (n_chunks == nullptr) return GCLIP_ERR_INVALID_ARG;
  std::vector<clip_chunk_t> chunks;
  const int rc = gclip::build_chunks(descs, n_tensors, chunks);
  if (rc != GCLIP_OK) return rc;
  *n_chunks = static_cast<int64_t>(chunks.size());
  if (out != nullptr) {
    if (capacity < static_cast<int64_t>(chunks.size())) return GCLIP_ERR_INVALID_ARG;
    if (!chunks.empty())
      std::memcpy(out, chunks.data(), chunks.size() * sizeof(clip_chunk_t));
  }
  return GCLIP_OK;
}

extern "C" const char* clip_status_string(int32_t code) {
  switch (code) {
    case GCLIP_OK: return "ok";
    case GCLIP_ERR_INVALID_ARG: return "invalid argument";
    case GCLIP_ERR_OOM: return "out of memory";
    case GCLIP_ERR_CUDA: return "CUDA error";
    case GCLIP_ERR_UNSUPPORTED: return "unsupported on this device";
    case GCLIP_ERR_TOO_LARGE: return "larger than the fixed no-allocation scratch allows";
    default: return "unknown status";
  }
}
