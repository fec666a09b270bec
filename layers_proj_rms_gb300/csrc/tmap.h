// TMA tensor maps of bf16 and fp32 tensors for the tensor-core kernels (the driver's
// cuTensorMapEncodeTiled, looked up once through the runtime).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace mhc {

// A `rank`-dimensional bf16 tensor (dims innermost first, byte strides of
// dims 1.. rank-1), box `box`, the given swizzle, 256-byte L2 promotion, zero
// fill outside the tensor.  False if the map cannot be encoded.
bool tmap_bf16(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
               const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle sw);

// A row-major [rows][cols] bf16 matrix, box [box_rows][box_cols].
inline bool tmap_bf16_2d(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
                         uint32_t box_rows, uint32_t box_cols, CUtensorMapSwizzle sw)
{
    const uint64_t dims[2] = {cols, rows};
    const uint64_t strides[1] = {cols * 2};
    const uint32_t box[2] = {box_cols, box_rows};
    return tmap_bf16(m, base, 2, dims, strides, box, sw);
}

// A row-major [rows][cols] fp32 matrix, box [box_rows][box_cols].
bool tmap_f32_2d(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                 uint32_t box_cols, CUtensorMapSwizzle sw);

}  // namespace mhc
