// tma_host.h -- host-side TMA tensor-map encoding used by the tensor-core kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace ssd {

// 4-D bf16 tensor map: dims/box innermost first, strides of dims 1..3 in
// bytes (multiples of 16), swizzle 128/64/32 bytes (or 0).  Out-of-bounds
// elements of a box read as zero.  Returns false if the driver rejects it.
bool encode_tmap_bf16_4d(CUtensorMap* out, const void* base, const uint64_t dims[4],
                         const uint64_t strides_bytes[3], const uint32_t box[4], int swizzle_bytes);

}  // namespace ssd
