// internal.hpp -- declarations shared by the host planner and the CUDA
// translation unit of the clipping library.  Not installed, not part of the
// C ABI.
#pragma once

#include <cstdint>
#include <vector>

#include "../../include/gclip.h"

namespace gclip {

int elem_size(int32_t dtype);
int validate_descs(const clip_tensor_desc_t* descs, int32_t n);
int build_chunks(const clip_tensor_desc_t* descs, int32_t n,
                 std::vector<clip_chunk_t>& out);

}  // namespace gclip
