// Host helpers of runtime.cu used by the library's other entry points.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "gf.h"

namespace gf {

// Device of the calling thread's current driver context (else the runtime's).
gf_status runtime_current_device(int* dev);

// The calling thread's current driver context (nullptr when there is none or
// the driver call is unavailable).
CUcontext runtime_current_context();

// Records `s` as the calling thread's last error (gf_last_error) and returns it.
gf_status runtime_fail(gf_status s);

// 2-D TMA map over a row-major [outer, inner] matrix of 16-bit elements with
// box_inner x box_outer boxes, 128-byte swizzle, zero fill out of bounds.
bool runtime_encode_2d(CUtensorMap* map, const void* ptr, gf_dtype dt, uint64_t inner,
                       uint64_t outer, uint32_t box_inner, uint32_t box_outer);

}  // namespace gf
