// Internal definitions shared by the library's translation units: the device
// segment table, launch helpers and small device utilities.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <vector>

#include "../../include/tf.h"

namespace tf {

// One stream's row of the device table (32 bytes).
struct SegStream {
    int32_t rows, row_offset, keys, cap;
    int32_t chunk_keys, n_chunks;
    int64_t pbase;            // first partial record of the stream
};

// A conv tile: up to 8 consecutive rows of one stream.
struct ConvTile {
    int32_t stream, row0, nrows, pad;
};

// An attention work item: one key chunk of one stream (for every KV head).
struct AttnItem {
    int32_t stream, chunk;
};

constexpr int kConvTileRows = 8;

// Device view of a segment table, passed to kernels by value.
struct SegTable {
    const SegStream* streams;
    const int32_t* row_stream;        // [R] stream of each row
    const ConvTile* tiles;            // [n_tiles]
    const AttnItem* items;            // [n_items], largest chunks first
    void* const* conv_state;          // [n_conv][S]
    void* const* conv_hist;           // [n_conv][S] or nullptr
    const void* const* k_cache;       // [n_attn][S]
    const void* const* v_cache;       // [n_attn][S]
    int32_t S, R, n_tiles, n_items, n_conv, n_attn, max_rows, has_hist;
    int64_t n_partials;
};

}  // namespace tf

// Host object behind the opaque tf_segments handle.
struct tf_segments {
    tf::SegTable dev;                  // pointers into `blob`
    void* blob = nullptr;              // one device allocation
    std::vector<unsigned char> host;   // host image of the blob (kept for the async copy)
    std::vector<tf::SegStream> streams;
    tf_plan plan{};
};

namespace tf {

// Record a CUDA error for tf_last_cuda_error and map it to TF_ECUDA.
int cuda_fail(cudaError_t e);

// Check the launch just issued.
inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TF_OK : cuda_fail(e);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Number of SMs of the current device (cached per device).
int sm_count();

// attn.cu: one attention layer's partials and merge with the records at po/pml.
int launch_attn_partials(const SegTable& t, int layer, const uint16_t* q, float* po, float2* pml,
                         cudaStream_t stream);
int launch_attn_merge(const SegTable& t, const float* po, const float2* pml, float* out, cudaStream_t stream);

}  // namespace tf
