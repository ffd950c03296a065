// a2/a3: causal GQA attention of every window row against its stream's KV
// cache, as split-K partials and a log-sum-exp merge, one launch each a layer.
//
// PR #1377 "LFM2: shared-round decode": commit "the conv, qk, attention and
// merge kernels' bodies as inline functions" (qk, attention, merge) and commit
// "a shared round runs each layer's conv and attention once over all its
// streams" (one launch a layer over every row from the segment table; the
// scratch's attention partials hold each stream's apart). PR #1391: the
// target's attention keeps its causal count.
//
// Partials kernel: one CTA per (work item = stream key chunk and group of at
// most 8 window rows, KV head). The chunk length depends on the stream alone
// (tf_chunk_keys: 256 * max(rows, 4) keys here), so a stream's partials do not
// depend on the other streams of the round. The CTA streams the chunk's K and
// V (64 keys a stage, 4-stage cp.async pipeline into XOR-swizzled shared
// memory) once, for the group's query rows of the KV head (GQA: query head h
// reads KV head h/4) -- a window of up to 8 rows shares one read of the
// cache; a wider one reads it once per group, the later groups from L2. The
// item's arithmetic (attn_item.cuh): four warps split each stage's keys, q.k
// on bf16 mma.sync with fp32 accumulation, P.V in fp16, and the item
// recomputed with V in bf16 (exact in V) when the fp16 pass left a partial
// sum that is not finite or every partial output below 2^-10.
//
// HBM bound: 256 bytes of K+V per key per KV head; the window's queries ride
// along. Arithmetic intensity 4*rows flops per byte for each of q.k and P.V.
//
// The same kernels serve the drafter's block attention (PR #1391: the
// target's attention and merge kernels under a FULL flag, with every row of a
// block seeing the keys [0, len + 1)): with `full` set every window row sees
// all of the stream's keys instead of its causal count; nothing else changes,
// and the merge is shared (it reads only the records).
#include "attn_item.cuh"

namespace tf {
namespace {

using item::kThreads;
using item::smem_bytes;
using item::ex2;

// One and two query m-tiles fit three CTAs per SM (<= 170 registers, 66 KB of
// smem each; measured 12% faster on 6-row windows than two CTAs). Wider
// windows run as several items of at most two m-tiles: a third m-tile needs
// 230 registers (two CTAs per SM), squeezed to three CTAs it spills, and
// either way the whole launch ran slower.
template <int MT>
__global__ void __launch_bounds__(kThreads, 3)
attn_partials_kernel(SegTable t, int layer, const uint16_t* __restrict__ q,
                     float* __restrict__ part_o, float2* __restrict__ part_ml, float* __restrict__ out,
                     int full) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int g = blockIdx.x % TF_NKV;
    const AttnItem it = t.items[blockIdx.x / TF_NKV];
    const SegStream st = t.streams[it.stream];
    if constexpr (MT == 1) {
        // narrow windows (one m-tile: short launches, one wave): the first
        // stages' keys and values into L2 while the previous kernel finishes
        // (measured 17.0 -> 16.0 us a layer for 16 one-row streams; the
        // two-m-tile kernel spilled with it and ran slower)
        if (threadIdx.x == 0) {
            const int c0 = it.chunk * st.chunk_keys;
            const int nkeys = min(st.chunk_keys, st.keys - c0);
            const size_t slot = size_t(layer) * t.S + it.stream;
            const size_t off = (size_t(g) * st.cap + c0) * TF_D;
            const uint32_t pre = uint32_t(min(nkeys, (item::kStages - 1) * item::kKT)) * item::kRowB;
            l2_prefetch_bulk(static_cast<const uint16_t*>(t.k_cache[slot]) + off, pre);
            l2_prefetch_bulk(static_cast<const uint16_t*>(t.v_cache[slot]) + off, pre);
        }
    }
    pdl_wait();   // the table above; queries and caches below
    const int mode = out ? st.merge_mode : kMergeKernel;   // records only in the two-call form
    item::attn_item<MT, true, 0>(t, layer, it, st, g, q, part_o, part_ml, out, mode, full, smem, threadIdx.x, true);
    if (mode == kMergeLastCta) {
        __shared__ int last_flag;
        finish_last_cta<MT == 1 ? 8 : 16>(t, layer, it.stream, st, g, part_o, part_ml, out, &last_flag);
    }
}

constexpr int kMergeSplit = 4;                       // warps per (row, query head)
constexpr int kMergeHeads = 2;                       // query heads per CTA
constexpr int kMergeThreads = kMergeSplit * kMergeHeads * 32;
constexpr int kMergeCtasPerRow = TF_NQ / kMergeHeads;
constexpr int kMergeLoads = 12;                      // 16-byte record loads in flight per lane
constexpr int kMergeBatch = 2 * kMergeLoads;         // records per warp batch (a half-warp reads one)

// kMergeSplit warps share one (row, query head): warp k takes the chunks
// c = k, k + kMergeSplit, ...; it reads them kMergeBatch at a time in one
// round trip: lane j the (m, l) of the batch's chunk j, and each half-warp
// every other chunk's o (lane holding dimensions 4*(lane%16) .. +3), all
// loads issued before any is used. The batch's weights take a running max
// (earlier batches rescaled when it grows). The warps' (M, L, o) are combined
// through shared memory at the end. 3 CTAs per SM: the long-context
// workload's 24 rows x 16 head pairs fit one wave.
__global__ void __launch_bounds__(kMergeThreads, 3)
attn_merge_kernel(SegTable t, const float* __restrict__ part_o, const float2* __restrict__ part_ml,
                  float* __restrict__ out, int kernel_mode_only) {
    const int row = blockIdx.x / kMergeCtasPerRow;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hl = warp / kMergeSplit, split = warp % kMergeSplit;
    const int h = (blockIdx.x % kMergeCtasPerRow) * kMergeHeads + hl;
    const int s = t.row_stream[row];
    const SegStream st = t.streams[s];
    if (kernel_mode_only && st.merge_mode != kMergeKernel) {   // finished by the partials kernel
        pdl_trigger();
        return;
    }
    const int i = row - st.row_offset;
    const int nq = st.rows * 4;
    const int g = h >> 2, hh = h & 3;
    const int64_t stride = int64_t(TF_NKV) * nq;   // records between chunks
    const int64_t base = st.pbase + int64_t(g) * nq + i * 4 + hh;
    const int C = st.n_chunks;
    const int nc = C > split ? (C - split + kMergeSplit - 1) / kMergeSplit : 0;   // this warp's chunks
    const int half = lane >> 4, d4 = (lane & 15) * 4;
    pdl_wait();

    // chunk j of this warp is c = split + j * kMergeSplit
    float M = -INFINITY;                              // running max over the batches so far
    float lsum = 0.f;                                 // this lane's share of the weight sum
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);     // dimensions d4.., chunks of parity `half`
    for (int j0 = 0; j0 < nc; j0 += kMergeBatch) {
        const int n = min(kMergeBatch, nc - j0);
        float2 ml = make_float2(-INFINITY, 0.f);
        if (lane < n) ml = part_ml[base + int64_t(split + (j0 + lane) * kMergeSplit) * stride];
        float4 v[kMergeLoads];
#pragma unroll
        for (int k = 0; k < kMergeLoads; ++k) {
            const int j = 2 * k + half;
            v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < n)
                v[k] = *reinterpret_cast<const float4*>(
                    part_o + (base + int64_t(split + (j0 + j) * kMergeSplit) * stride) * TF_D + d4);
        }
        float mb = ml.y > 0.f ? ml.x : -INFINITY;   // empty partials (l = 0) carry no weight
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, o));
        const float Mn = fmaxf(M, mb);
        if (Mn == -INFINITY) continue;               // nothing visible yet (warp-uniform)
        if (M != -INFINITY && Mn > M) {
            const float f = ex2(M - Mn);
            lsum *= f;
            acc.x *= f;
            acc.y *= f;
            acc.z *= f;
            acc.w *= f;
        }
        M = Mn;
        const float wj = ml.y > 0.f ? ex2(ml.x - M) : 0.f;
        lsum += wj * ml.y;
#pragma unroll
        for (int k = 0; k < kMergeLoads; ++k) {
            const float wk = __shfl_sync(0xFFFFFFFFu, wj, 2 * k + half);
            acc.x += wk * v[k].x;
            acc.y += wk * v[k].y;
            acc.z += wk * v[k].z;
            acc.w += wk * v[k].w;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, o);
    acc.x += __shfl_xor_sync(0xFFFFFFFFu, acc.x, 16);   // the two halves' chunks
    acc.y += __shfl_xor_sync(0xFFFFFFFFu, acc.y, 16);
    acc.z += __shfl_xor_sync(0xFFFFFFFFu, acc.z, 16);
    acc.w += __shfl_xor_sync(0xFFFFFFFFu, acc.w, 16);
    pdl_trigger();

    // combine the kMergeSplit warps of each head
    __shared__ float sM[kMergeHeads][kMergeSplit], sL[kMergeHeads][kMergeSplit];
    __shared__ float4 sO[kMergeHeads][kMergeSplit][16];
    if (lane == 0) {
        sM[hl][split] = M;
        sL[hl][split] = lsum;
    }
    if (lane < 16) sO[hl][split][lane] = acc;
    __syncthreads();
    if (split == 0 && lane < 16) {
        float Mt = -INFINITY;
#pragma unroll
        for (int k = 0; k < kMergeSplit; ++k) Mt = fmaxf(Mt, sM[hl][k]);
        float L = 0.f;
        float4 o4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < kMergeSplit; ++k) {
            if (sM[hl][k] == -INFINITY) continue;   // no visible key in this warp's chunks
            const float f = ex2(sM[hl][k] - Mt);
            L += f * sL[hl][k];
            const float4 w4 = sO[hl][k][lane];
            o4.x += f * w4.x;
            o4.y += f * w4.y;
            o4.z += f * w4.z;
            o4.w += f * w4.w;
        }
        const float inv = 1.f / L;
        *reinterpret_cast<float4*>(out + (size_t(row) * TF_NQ + h) * TF_D + d4) =
            make_float4(o4.x * inv, o4.y * inv, o4.z * inv, o4.w * inv);
    }
}

template <int MT>
int prepare_one() {
    cudaError_t e = cudaFuncSetAttribute(attn_partials_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes(MT));
    return e == cudaSuccess ? TF_OK : cuda_fail(e);
}

}  // namespace

int attn_prepare() {
    int rc;
    if ((rc = prepare_one<1>()) != TF_OK) return rc;
    return prepare_one<2>();
}

// Launchers for other translation units: the partials and the merge of one
// attention layer with the partial records at `po` (o) and `pml` (m, l).
int launch_attn_partials(const SegTable& t, int layer, const uint16_t* q, float* po, float2* pml,
                         cudaStream_t stream, float* out, int full) {
    if (t.n_items_mma > 0 && t.n_items_mma < t.n_items && t.side) {
        // both kinds of windows: the two launches run side by side (they write
        // disjoint streams' records and outputs). The persistent tensor-core
        // grid, sized to its share of the keys, stays on the caller's stream,
        // where it launches early (programmatic dependent launch) and holds its
        // SMs; the mma.sync launch, forked onto the table's side stream, fills
        // the rest once the previous kernel is done. (The other way round the
        // early mma.sync launch took every SM before the tensor-core one.)
        cudaError_t e = cudaEventRecord(t.ev_fork, stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(t.side, t.ev_fork, 0);
        if (e != cudaSuccess) return cuda_fail(e);
        int rc = launch_attn_partials_tc(t, layer, q, po, pml, stream, out, full, t.tc_grid_mixed);
        if (rc != TF_OK) return rc;
        const dim3 grid(t.n_items_mma * TF_NKV);
        if (t.mma_mt == 1)
            rc = launch_pdl(attn_partials_kernel<1>, grid, dim3(kThreads), smem_bytes(1), t.side, t, layer, q, po, pml,
                            out, full);
        else
            rc = launch_pdl(attn_partials_kernel<2>, grid, dim3(kThreads), smem_bytes(2), t.side, t, layer, q, po, pml,
                            out, full);
        if (rc != TF_OK) return rc;
        e = cudaEventRecord(t.ev_join, t.side);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, t.ev_join, 0);
        return e == cudaSuccess ? TF_OK : cuda_fail(e);
    }
    if (t.n_items_mma > 0) {
        const dim3 grid(t.n_items_mma * TF_NKV);
        int rc;
        if (t.mma_mt == 1)
            rc = launch_pdl(attn_partials_kernel<1>, grid, dim3(kThreads), smem_bytes(1), stream, t, layer, q, po, pml,
                            out, full);
        else
            rc = launch_pdl(attn_partials_kernel<2>, grid, dim3(kThreads), smem_bytes(2), stream, t, layer, q, po, pml,
                            out, full);
        if (rc != TF_OK) return rc;
    }
    if (t.n_items_mma < t.n_items) return launch_attn_partials_tc(t, layer, q, po, pml, stream, out, full);
    return TF_OK;
}

int launch_attn_merge(const SegTable& t, const float* po, const float2* pml, float* out, cudaStream_t stream,
                      bool kernel_mode_only) {
    return launch_pdl(attn_merge_kernel, dim3(t.R * kMergeCtasPerRow), dim3(kMergeThreads), 0, stream, t, po, pml,
                      out, kernel_mode_only ? 1 : 0);
}

}  // namespace tf

extern "C" int tf_attn_partials(const tf_segments* seg, int attn_layer, const void* q, void* partials,
                                tf_cuda_stream stream) {
    using namespace tf;
    if (!seg) return TF_EINVAL;
    const SegTable& t = seg->dev;
    if (attn_layer < 0 || attn_layer >= t.n_attn) return TF_EINVAL;
    if (t.R == 0) return TF_OK;
    if (!q || !partials || !aligned16(q) || !aligned16(partials)) return TF_EINVAL;
    float* po = static_cast<float*>(partials);
    float2* pml = reinterpret_cast<float2*>(po + t.n_partials * TF_D);
    return launch_attn_partials(t, attn_layer, static_cast<const uint16_t*>(q), po, pml, stream);
}

extern "C" int tf_attn(const tf_segments* seg, int attn_layer, const void* q, void* partials, float* out,
                       tf_cuda_stream stream) {
    using namespace tf;
    if (!seg) return TF_EINVAL;
    const SegTable& t = seg->dev;
    if (attn_layer < 0 || attn_layer >= t.n_attn) return TF_EINVAL;
    if (t.R == 0) return TF_OK;
    if (!q || !partials || !out || !aligned16(q) || !aligned16(partials) || !aligned16(out)) return TF_EINVAL;
    float* po = static_cast<float*>(partials);
    float2* pml = reinterpret_cast<float2*>(po + t.n_partials * TF_D);
    int rc = launch_attn_partials(t, attn_layer, static_cast<const uint16_t*>(q), po, pml, stream, out);
    if (rc != TF_OK || t.n_merge_rows == 0) return rc;
    return launch_attn_merge(t, po, pml, out, stream, true);
}

extern "C" int tf_attn_block_partials(const tf_segments* seg, int attn_layer, const void* q, void* partials,
                                      tf_cuda_stream stream) {
    using namespace tf;
    if (!seg) return TF_EINVAL;
    const SegTable& t = seg->dev;
    if (attn_layer < 0 || attn_layer >= t.n_attn) return TF_EINVAL;
    if (t.R == 0) return TF_OK;
    if (!q || !partials || !aligned16(q) || !aligned16(partials)) return TF_EINVAL;
    float* po = static_cast<float*>(partials);
    float2* pml = reinterpret_cast<float2*>(po + t.n_partials * TF_D);
    return launch_attn_partials(t, attn_layer, static_cast<const uint16_t*>(q), po, pml, stream, nullptr, 1);
}

extern "C" int tf_attn_block(const tf_segments* seg, int attn_layer, const void* q, void* partials, float* out,
                             tf_cuda_stream stream) {
    using namespace tf;
    if (!seg) return TF_EINVAL;
    const SegTable& t = seg->dev;
    if (attn_layer < 0 || attn_layer >= t.n_attn) return TF_EINVAL;
    if (t.R == 0) return TF_OK;
    if (!q || !partials || !out || !aligned16(q) || !aligned16(partials) || !aligned16(out)) return TF_EINVAL;
    float* po = static_cast<float*>(partials);
    float2* pml = reinterpret_cast<float2*>(po + t.n_partials * TF_D);
    int rc = launch_attn_partials(t, attn_layer, static_cast<const uint16_t*>(q), po, pml, stream, out, 1);
    if (rc != TF_OK || t.n_merge_rows == 0) return rc;
    return launch_attn_merge(t, po, pml, out, stream, true);
}

extern "C" int tf_attn_merge(const tf_segments* seg, const void* partials, float* out, tf_cuda_stream stream) {
    using namespace tf;
    if (!seg) return TF_EINVAL;
    const SegTable& t = seg->dev;
    if (t.R == 0) return TF_OK;
    if (!partials || !out || !aligned16(partials) || !aligned16(out)) return TF_EINVAL;
    const float* po = static_cast<const float*>(partials);
    const float2* pml = reinterpret_cast<const float2*>(po + t.n_partials * TF_D);
    return launch_attn_merge(t, po, pml, out, stream, false);
}
