// Internal definitions shared by the library's translation units: the device
// segment table, launch helpers and small device utilities.
#pragma once

#include <cuda.h>            // CUtensorMap (the type only; the encoder comes from the runtime's driver entry point)
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
    int32_t merge_mode;       // in one-call attention: kMergeDirect / kMergeLastCta / kMergeKernel
    int32_t n_qg;             // query groups: items per key chunk (mma.sync path: one per 8 window rows)
};

// How the one-call attention (tf_attn) finishes a stream's chunks.
constexpr int kMergeDirect = 0;    // one chunk: the partials kernel writes the output
constexpr int kMergeLastCta = 1;   // few records: the last CTA of each KV head merges them
constexpr int kMergeKernel = 2;    // many records: the merge kernel
constexpr int kMergeLastCtaMaxRecords = 512;   // 4*rows*chunks of one KV head

// A conv tile: up to 8 consecutive rows of one stream.
struct ConvTile {
    int32_t stream, row0, nrows, pad;
};

// An attention work item: one key chunk of one stream (for every KV head) and,
// on the mma.sync path, one group of at most kMmaGroupRows window rows: query
// rows [q0, q0 + 4*kMmaGroupRows) of the KV head (q0 = 0 on the tensor-core
// path, which takes the whole window).
struct AttnItem {
    int32_t stream, chunk, q0, pad;
};

// Window rows of one mma.sync item: two 16-row query m-tiles, the most that
// keep three CTAs per SM. Wider windows run as several items over the same
// chunk, next to each other in the grid (the second read of the chunk comes
// from L2).
constexpr int kMmaGroupRows = 8;

constexpr int kConvTileRows = 8;
// A prompt call's attention runs in windows of this many rows: 32 rows x 4
// query heads fill the 128 TMEM lanes of a tcgen05 tile (16-row tiles, those
// of the per-stream kernels, fill half of it).
constexpr int kPromptTileRows = TF_PROMPT_WINDOW_ROWS;

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
    const CUtensorMap* k_maps;        // [n_attn][S] TMA maps of the K caches (tensor-core path)
    const CUtensorMap* v_maps;        // [n_attn][S]
    int32_t S, R, n_tiles, n_items, n_conv, n_attn, max_rows, has_hist;
    int32_t n_items_mma;              // items [0, n_items_mma) run on the mma.sync kernel,
                                      // [n_items_mma, n_items) on the tcgen05 kernel
    int32_t mma_mt;                   // 16-row query tiles of the mma.sync kernel's widest item (1 or 2)
    int64_t n_partials;
    int32_t* counters;                // [n_attn][S][8] arrivals per (stream, KV head), self-resetting
    int32_t n_merge_rows;             // rows of kMergeKernel streams
    int32_t pad2_;
    unsigned long long* mk_keys;      // [S] Markov step: best (score, token) key per stream, self-resetting
    uint32_t* mk_flags;               // [S] Markov step: nonfinite / gave-up bits per stream, self-resetting
    uint32_t* mk_ctr;                 // [ceil(S/128)] Markov step: CTA arrivals per stream group
    int32_t* tc_work;                 // [n_attn][2] tensor-core attention: units handed out, CTAs done (self-resetting)
    uint32_t* mk_sync;                // Markov chain in one launch (kMkSyncBytes, zeroed per launch): [0] arrivals,
                                      // [1] generation, [2] abort; from word 64 the per-step flags and keys
    int32_t* tc_redo;                 // tensor-core attention: [0] units queued for the exact recompute, [1..] them
    uint32_t* status;                 // TF_STATUS_* bits: a kernel gave up a bounded wait (tf_segments_status)
    unsigned long long wait_ns;       // limit of a device wait, set per launch from tf_set_wait_limit_ns
    // Host side only (no kernel reads them): a round holding both kinds of
    // attention windows runs its tensor-core launch on `side`, forked from and
    // joined back to the caller's stream, so that it runs alongside the
    // mma.sync launch; tc_grid_mixed is its grid then (its share of the keys).
    cudaStream_t side;
    cudaEvent_t ev_fork, ev_join;
    int32_t tc_grid_mixed;
    int32_t pad3_;
};

// The Markov chain's scratch: 64 words of barrier state, then three
// generations of 64 flag words (from word 64) and of 8 x 64 keys (from byte 1024).
constexpr int kMkSyncBytes = 1024 + 3 * 8 * 64 * 8;

constexpr int kAttnMma = 0;   // mma.sync flash-decode kernel (narrow windows)
constexpr int kAttnTc = 1;    // tcgen05 + TMA kernel (windows of 9 rows or more)
// Measured on GB300: the mma.sync kernel streams faster up to 8-row windows
// (one item); from 9 rows, where mma.sync takes a window as two items of at
// most 8 rows that read the chunk twice, the tensor-core kernel wins (one unit
// reads it once: 64 streams of U{1..16} rows 1,403 -> 1,280 us a step).
constexpr int kTcMinRows = 9;

// Kernel of a stream: by its window rows, unless TF_ATTN_PATH forces one.
int attn_path_of(int rows);

// segments.cu: TMA map of a bf16 [rows][256] matrix (the Markov head's W2),
// boxes of 128 rows x 64 columns with 128-byte swizzle; rows past `rows` read
// as zeros. False when the driver refuses it.
bool encode_w2_map(CUtensorMap* out, const void* w2, int rows);
// segments.cu: TMA map of the queries bf16 [rows][TF_NQ][TF_D] as (d, head, row),
// boxes of 4 heads x 4 rows (16 query rows of one KV head's group), 128-byte
// swizzle; rows past `rows` read as zeros. False when the driver refuses it.
bool encode_q_map(CUtensorMap* out, const void* q, int rows);

}  // namespace tf

// Host object behind the opaque tf_segments handle.
struct tf_segments {
    tf::SegTable dev;                  // pointers into `blob`
    void* blob = nullptr;              // one device allocation
    std::vector<unsigned char> host;   // host image of the blob (kept for the async copy)
    std::vector<tf::SegStream> streams;
    tf_plan plan{};
    bool prompt = false;               // built by tf_prompt_build (conv + attention only)
    size_t scratch_off = 0;            // the blob's cross-CTA scratch and status word:
    size_t scratch_bytes = 0;          // zero in the image, zeroed again by tf_segments_status
};

namespace tf {

// Record a CUDA error for tf_last_cuda_error and map it to TF_ECUDA.
int cuda_fail(cudaError_t e);

// The current limit of a device wait (tf_set_wait_limit_ns), in nanoseconds.
unsigned long long wait_limit_ns();

// Check the launch just issued.
inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TF_OK : cuda_fail(e);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Number of SMs of the current device (cached per device).
int sm_count();

// ---- programmatic dependent launch ---------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialization: it may start while the previous kernel of the stream is
// finishing. Before griddepcontrol.wait a kernel reads nothing but the
// segment table (immutable once built, uploaded before any launch that uses
// it) and may issue L2 prefetches (l2_prefetch_bulk); after it, everything
// the previous kernels wrote is visible. Each kernel
// lets its dependents launch once it has finished its main work.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Bulk prefetch of [p, p + bytes) into L2 (16-byte aligned, bytes a multiple
// of 16). A non-binding hint, so a kernel may issue it before pdl_wait: L2 is
// the GPU's point of coherence, and a line a previous kernel is still writing
// is not read into the kernel early.
__device__ __forceinline__ void l2_prefetch_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
               Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    if (e != cudaSuccess) return cuda_fail(e);
    return launch_status();
}

// attn.cu: one attention layer's partials and merge with the records at po/pml.
// With out != nullptr the partials kernels also finish the streams whose
// merge_mode is kMergeDirect or kMergeLastCta (the one-call form). full != 0:
// the drafter's non-causal block form, every window row seeing all keys.
int launch_attn_partials(const SegTable& t, int layer, const uint16_t* q, float* po, float2* pml,
                         cudaStream_t stream, float* out = nullptr, int full = 0);
int launch_attn_merge(const SegTable& t, const float* po, const float2* pml, float* out, cudaStream_t stream,
                      bool kernel_mode_only = false);

// attn_tc.cu: the tensor-core partials kernel (same records as the mma.sync kernel).
int launch_attn_partials_tc(const SegTable& t, int layer, const uint16_t* q, float* po, float2* pml,
                            cudaStream_t stream, float* out, int full,
                            int grid = 0);   // items [n_items_mma, n_items); grid 0: two CTAs per SM
int attn_tc_prepare();

}  // namespace tf

namespace tf {

// ---- shared device code of the attention kernels -------------------------

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Largest |v| of two bf16 pairs, per half (the sign bits of the result are
// not meaningful; NaN inputs are ignored).
__device__ __forceinline__ uint32_t absmax_bf2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// Whether a V tile with largest magnitude bits `m` (|v| as a bf16 bit
// pattern) takes the exact bf16 path of P.V: |v| of 65,536 or more has no
// fp16 value (fp16's largest is 65,504), and a tile whose values all lie
// below 2^-6 would lose relative precision to fp16's subnormals (steps of
// 2^-24). Any other tile converts to fp16 with an absolute error of at most
// 2^-25 per value (only values below 2^-14 round at all).
__device__ __forceinline__ bool v_tile_exact(uint32_t m) { return m >= 0x4780u || m < 0x3C80u; }

// Output address of query row qi (window row qi/4, head 4g + qi%4) of a stream.
__device__ __forceinline__ float* out_row(float* out, const SegStream& st, int g, int qi) {
    return out + (size_t(st.row_offset + (qi >> 2)) * TF_NQ + 4 * g + (qi & 3)) * TF_D;
}

// Log-sum-exp merge of the chunk records of one (stream, KV head) into the
// output, by the threads [tid, nthreads) of one CTA, one pass over the chunks
// kB at a time with a running max. A thread takes kU of its (query row, 4
// dimensions) items at once and issues all their loads before using any
// (kU = 1: one item at a time). The records were written by other CTAs: they
// are read through L2 (ld.global.cg).
template <int kB, int kU = 1>   // records in flight per item, items per thread at once
__device__ __forceinline__ void merge_stream_head(const SegStream& st, int g, const float* part_o,
                                                  const float2* part_ml, float* out, int tid, int nthreads) {
    const int nq = st.rows * 4;
    const int n_items = nq * (TF_D / 4);
    const int64_t stride = int64_t(TF_NKV) * nq;
    const int64_t base = st.pbase + int64_t(g) * nq;
    for (int i0 = tid; i0 < n_items; i0 += nthreads * kU) {
        float M[kU], L[kU];
        float4 acc[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            M[u] = -INFINITY;
            L[u] = 0.f;
            acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int c0 = 0; c0 < st.n_chunks; c0 += kB) {
            float2 ml[kU][kB];
            float4 v[kU][kB];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int idx = i0 + u * nthreads;
                const int qi = idx >> 4, d4 = (idx & 15) * 4;
#pragma unroll
                for (int k = 0; k < kB; ++k) {
                    ml[u][k] = make_float2(-INFINITY, 0.f);
                    v[u][k] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (idx < n_items && c0 + k < st.n_chunks) {
                        const int64_t rec = base + (c0 + k) * stride + qi;
                        ml[u][k] = __ldcg(part_ml + rec);
                        v[u][k] = __ldcg(reinterpret_cast<const float4*>(part_o + rec * TF_D + d4));
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                float Mb = M[u];
#pragma unroll
                for (int k = 0; k < kB; ++k)
                    if (ml[u][k].y > 0.f) Mb = fmaxf(Mb, ml[u][k].x);
                if (Mb == -INFINITY) continue;
                const float sc = (M[u] == -INFINITY) ? 0.f : ex2_approx(M[u] - Mb);
                L[u] *= sc;
                acc[u].x *= sc;
                acc[u].y *= sc;
                acc[u].z *= sc;
                acc[u].w *= sc;
                M[u] = Mb;
#pragma unroll
                for (int k = 0; k < kB; ++k) {
                    if (ml[u][k].y > 0.f) {
                        const float w = ex2_approx(ml[u][k].x - Mb);
                        L[u] += w * ml[u][k].y;
                        acc[u].x += w * v[u][k].x;
                        acc[u].y += w * v[u][k].y;
                        acc[u].z += w * v[u][k].z;
                        acc[u].w += w * v[u][k].w;
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int idx = i0 + u * nthreads;
            if (idx < n_items) {
                const int qi = idx >> 4, d4 = (idx & 15) * 4;
                const float inv = 1.f / L[u];
                *reinterpret_cast<float4*>(out_row(out, st, g, qi) + d4) =
                    make_float4(acc[u].x * inv, acc[u].y * inv, acc[u].z * inv, acc[u].w * inv);
            }
        }
    }
}

// End of a partials CTA in the one-call form, for kMergeLastCta streams: every
// CTA of (stream, KV head) counts its arrival after its records are visible;
// the last one merges and resets the counter for the next launch. All threads
// of the CTA call this.
template <int kB = 8>
__device__ __forceinline__ void finish_last_cta(const SegTable& t, int layer, int s, const SegStream& st, int g,
                                                const float* part_o, const float2* part_ml, float* out,
                                                int* smem_flag) {
    __threadfence();
    __syncthreads();
    int* ctr = t.counters + (size_t(layer) * t.S + s) * TF_NKV + g;
    if (threadIdx.x == 0) *smem_flag = (atomicAdd(ctr, 1) == st.n_chunks * st.n_qg - 1);
    __syncthreads();
    if (*smem_flag) {
        __threadfence();
        merge_stream_head<kB>(st, g, part_o, part_ml, out, threadIdx.x, blockDim.x);
        if (threadIdx.x == 0) atomicExch(ctr, 0);
    }
}

}  // namespace tf
