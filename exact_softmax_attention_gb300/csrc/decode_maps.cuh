// Tensor-map form of the 8-bit paged decode (interface between attn_api.cu and attn_decode.cu).
#pragma once

#include "kernels.cuh"

namespace attn {

// 2-D maps over the 8-bit key and value caches viewed as [num_pages * page_size rows, Hkv * d
// bytes]; box d bytes x 16 rows, 128-byte swizzle. When the page size is a multiple of 16, the 16
// tokens of a split kernel's token group lie in one page, so one map load brings the group's K
// (or V) rows of one kv head.
struct DecodeTmaps {
    CUtensorMap k, v;
};

// Rows of one map load (tokens of a token group).
constexpr int kDecodeMapRows = 16;

// As launch_attn_decode_fp8, with the K/V rows of each token group loaded through the maps
// (d = 128, page_size % 16 == 0; other shapes are cudaErrorInvalidValue).
cudaError_t launch_attn_decode_fp8_maps(const DecodeParams& p, const DecodeTmaps& tm, int d, int fmt,
                                        cudaStream_t stream);

}  // namespace attn
