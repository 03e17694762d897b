// Host helper: tensor maps for the tensor-memory accelerator (TMA) over bf16 activations, encoded
// through the driver entry point that the CUDA runtime exposes (no link against libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rapt {

// Tiled bf16 map of `rank` (<= 5) dimensions, innermost first: dims[i] elements, strides[i] bytes
// between consecutive indices of dimension i + 1 (multiples of 16), box[i] elements per copy.
// 128-byte swizzle (box[0] * 2 must be 128), zero fill outside the tensor. Returns
// cudaErrorNotSupported if the driver entry point is missing, cudaErrorInvalidValue if the driver
// rejects the description (base not 16-byte aligned, bad strides or box).
cudaError_t encode_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                            const uint64_t* strides, const uint32_t* box);

// [rows, H, D] (rows = B * L or T): boxes of 64 x 1 x 128 (one 64-column block of a 128-row tile).
cudaError_t make_rows_map(CUtensorMap* map, const void* base, long rows, int H, int D);

// [B, L, H, D]: boxes of 64 x 1 x 128 x 1; rows past L read as zero and are not written by stores,
// so a tile at the end of one batch row never touches the next.
cudaError_t make_bshd_map(CUtensorMap* map, const void* base, int B, int L, int H, int D);

}  // namespace rapt
