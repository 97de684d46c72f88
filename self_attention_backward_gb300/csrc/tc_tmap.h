// tc_tmap.h -- host-side TMA tensor-map encoding shared by the tensor-core
// translation units.
#pragma once

#include <cuda.h>

#include <string>

namespace psa {

// 3-D tiled map over a bf16 tensor laid out as Z slices of [N, D] rows (row
// stride D elements, slice stride N*D), copied in boxes of `rows` rows by
// `cols` columns (cols <= D, cols*2 bytes a multiple of 16); the shared-memory
// swizzle span equals the box's row bytes (128, 64 or 32).  Rows past N are
// out of bounds and read as zeros.  Returns false and sets *err on failure.
bool encode_bf16_rows(CUtensorMap* map, const void* base, int D, int N, long long Z, int rows, int cols,
                      std::string* err);
// The same with rows `ld` elements apart (ld >= D, ld * 2 a multiple of 16).
bool encode_bf16_rows_ld(CUtensorMap* map, const void* base, int D, long long ld, int N, long long Z, int rows,
                         int cols, std::string* err);
// 4-D map over a bf16 tensor [B][heads][outer][inner] with element strides
// 1, s_outer, s_head, s_batch (each but the first a multiple of 8), copied in
// boxes of box_inner x box_outer (box_inner * 2 bytes = 32, 64 or 128, the
// swizzle span); elements past the extents read as zeros.
bool encode_bf16_4d(CUtensorMap* map, const void* base, long long inner, long long outer, long long heads,
                    long long B, long long s_outer, long long s_head, long long s_batch, int box_inner,
                    int box_outer, std::string* err);

// The same over an fp32 tensor of Z slices of [N, D] rows, boxes of `rows` x
// `cols` (cols * 4 bytes a multiple of 16, at most 128; the swizzle span is the
// box's row bytes: 128, 64 or 32).
bool encode_f32_rows(CUtensorMap* map, const void* base, int D, int N, long long Z, int rows, int cols,
                     std::string* err);

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device) pair for the life of the process (a
// function attribute is per device, so a second GPU needs its own call).
// Returns false and sets *err on failure.
bool set_max_dynamic_smem(const void* kernel, int bytes, std::string* err);

// 1 if the dynamic shared memory of a kernel without static shared memory
// starts on a 1024-byte boundary on the current device (kernels whose 128B-
// swizzled layout fills shared memory leave no room to align it themselves),
// 0 if not, -1 on a CUDA error (*err set).  A one-thread probe kernel, run
// once per device on a private stream.
int dyn_smem_base_aligned(std::string* err);

}  // namespace psa
