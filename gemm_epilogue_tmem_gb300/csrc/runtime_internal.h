// Host helpers of runtime.cu used by the library's other entry points.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "gf.h"

namespace gf {

// Device of the calling thread's current driver context (else the runtime's).
gf_status runtime_current_device(int* dev);

// 2-D TMA map over a row-major [outer, inner] matrix of 16-bit elements with
// box_inner x box_outer boxes, 128-byte swizzle, zero fill out of bounds.
bool runtime_encode_2d(CUtensorMap* map, const void* ptr, gf_dtype dt, uint64_t inner,
                       uint64_t outer, uint32_t box_inner, uint32_t box_outer);

}  // namespace gf
