// a4: greedy pick over each row of bf16 logits.
//
// PR #1377 "LFM2: shared-round decode", commit "a verify's greedy rows take
// the GPU's pick of their logits": each row's largest logit is picked, the
// lowest id winning among equal values, and a row holding a nonfinite logit
// is flagged; the
// host used to scan the 128,000 bf16 logits of every row with the GPU idle.
//
// Design: a row is split over a thread-block cluster of `cl` CTAs (cl = 1..8,
// chosen so the grid fills the GPU even for a few rows). Each thread streams
// 16-byte vectors of its range in increasing id order and keeps the first
// largest value it met; per vector it takes the packed bf16x2 maximum and only
// searches the 8 lanes when that maximum beats the running best, which is rare.
// Nonfinite values are found from the exponent field (all ones). Threads, then
// warps, then CTAs are reduced by (value desc, id asc); the CTAs of a cluster
// meet in distributed shared memory, so the kernel needs no global scratch.
// HBM bound: 2 bytes per logit.
#include <cooperative_groups.h>

#include "tf_internal.cuh"

namespace cg = cooperative_groups;

namespace tf {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

struct Best {
    float v;
    int id;
};

// true when (v1, i1) comes before (v2, i2): larger value, then lower id
__device__ __forceinline__ bool better(float v1, int i1, float v2, int i2) {
    return v1 > v2 || (v1 == v2 && i1 < i2);
}

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Exponent field all ones (NaN or infinity) in either half sets bit 15 / 31.
__device__ __forceinline__ uint32_t nonfinite_bits(uint32_t w) {
    return (w & 0x7F807F80u) + 0x00800080u;
}

__device__ __forceinline__ void scan_vec(const uint4& v, int id0, float& best, int& bid, uint32_t& nf) {
    nf |= nonfinite_bits(v.x) | nonfinite_bits(v.y) | nonfinite_bits(v.z) | nonfinite_bits(v.w);
    __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&v.x),
                               *reinterpret_cast<const __nv_bfloat162*>(&v.y));
    __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&v.z),
                               *reinterpret_cast<const __nv_bfloat162*>(&v.w));
    __nv_bfloat162 m = __hmax2(a, b);
    const float mx = fmaxf(__bfloat162float(m.x), __bfloat162float(m.y));
    if (mx > best) {   // first lane holding mx (-0 == +0 under float compare)
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        int k = 7;
#pragma unroll
        for (int j = 7; j >= 0; --j) {
            const float f = (j & 1) ? hi_f(w[j >> 1]) : lo_f(w[j >> 1]);
            if (f == mx) k = j;
        }
        best = mx;
        bid = id0 + k;
    }
}

__device__ __forceinline__ void scan_one(uint16_t bits, int id, float& best, int& bid, uint32_t& nf) {
    nf |= ((uint32_t(bits) & 0x7F80u) + 0x0080u);
    const float f = __uint_as_float(uint32_t(bits) << 16);
    if (f > best) {
        best = f;
        bid = id;
    }
}

template <bool kVec>
__global__ void __launch_bounds__(kThreads)
argmax_rows_kernel(const uint16_t* __restrict__ logits, int V, int64_t stride, int chunk,
                   int32_t* __restrict__ pick, uint8_t* __restrict__ flag) {
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = int(cluster.block_rank());
    const int ncl = int(cluster.num_blocks());
    const int row = blockIdx.y;
    const uint16_t* p = logits + size_t(row) * size_t(stride);
    const int begin = rank * chunk;
    const int end = min(V, begin + chunk);

    float best = -INFINITY;
    int bid = 0x7FFFFFFF;
    uint32_t nf = 0;
    pdl_wait();

    if (kVec) {
        // vector part: [begin, vend), begin and chunk are multiples of 8
        const int vend = begin + ((max(end - begin, 0)) & ~7);
        const uint4* pv = reinterpret_cast<const uint4*>(p + begin);
        const int nvec = (vend - begin) >> 3;
        int i = threadIdx.x;
        for (; i + (kUnroll - 1) * kThreads < nvec; i += kUnroll * kThreads) {
            uint4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) v[u] = __ldcs(pv + i + u * kThreads);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) scan_vec(v[u], begin + 8 * (i + u * kThreads), best, bid, nf);
        }
        for (; i < nvec; i += kThreads) scan_vec(__ldcs(pv + i), begin + 8 * i, best, bid, nf);
        for (int j = vend + threadIdx.x; j < end; j += kThreads) scan_one(p[j], j, best, bid, nf);
    } else {
        for (int j = begin + threadIdx.x; j < end; j += kThreads) scan_one(p[j], j, best, bid, nf);
    }
    pdl_trigger();
    if (best == 0.0f) best = 0.0f;   // -0 -> +0 so keys compare as values
    bool bad = (nf & 0x80008000u) != 0;

    // warp, then CTA
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        const int i2 = __shfl_xor_sync(0xFFFFFFFFu, bid, o);
        if (better(v2, i2, best, bid)) {
            best = v2;
            bid = i2;
        }
    }
    bad = __any_sync(0xFFFFFFFFu, bad);
    __shared__ Best warp_best[kThreads / 32];
    __shared__ int warp_bad[kThreads / 32];
    __shared__ Best cta_best;
    __shared__ int cta_bad;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        warp_best[warp] = {best, bid};
        warp_bad[warp] = bad;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        Best b = warp_best[0];
        int any = warp_bad[0];
        for (int k = 1; k < kThreads / 32; ++k) {
            if (better(warp_best[k].v, warp_best[k].id, b.v, b.id)) b = warp_best[k];
            any |= warp_bad[k];
        }
        cta_best = b;
        cta_bad = any;
    }
    // the cluster's CTAs meet in distributed shared memory
    cluster.sync();
    if (rank == 0 && threadIdx.x == 0) {
        Best b = cta_best;
        int any = cta_bad;
        for (int r = 1; r < ncl; ++r) {
            const Best* ob = cluster.map_shared_rank(&cta_best, r);
            const int* oa = cluster.map_shared_rank(&cta_bad, r);
            const Best o = *ob;
            if (better(o.v, o.id, b.v, b.id)) b = o;
            any |= *oa;
        }
        pick[row] = any ? -1 : b.id;
        flag[row] = any ? 1 : 0;
    }
    cluster.sync();   // keep every CTA's shared memory alive until rank 0 has read it
}

}  // namespace
}  // namespace tf

extern "C" int tf_argmax_rows(const void* logits, int R, int V, int64_t row_stride,
                              int32_t* pick, uint8_t* flag, tf_cuda_stream stream) {
    using namespace tf;
    if (R < 0) return TF_EINVAL;
    if (R == 0) return TF_OK;
    if (!logits || !pick || !flag || V < 1 || row_stride < V) return TF_EINVAL;
    if (V > (1 << 30) || R > (1 << 24)) return TF_ERANGE;
    const bool vec = aligned16(logits) && (row_stride % 8) == 0;
    // CTAs per row: enough to fill every SM about 8 CTAs deep, at most 8
    const int target = sm_count() * 8;
    int cl = (target + R - 1) / R;
    cl = cl < 1 ? 1 : (cl > 8 ? 8 : cl);
    const int vecs = (V + 7) / 8;
    int chunk = ((vecs + cl - 1) / cl) * 8;
    cl = (V + chunk - 1) / chunk;   // no empty CTA
    if (cl < 1) cl = 1;

    // rows go in grid.y, at most 65,535 a launch: larger R takes several launches
    constexpr int kRowsPerLaunch = 65535;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see tf_internal.cuh
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    for (int r0 = 0; r0 < R; r0 += kRowsPerLaunch) {
        const int nr = R - r0 < kRowsPerLaunch ? R - r0 : kRowsPerLaunch;
        cfg.gridDim = dim3(cl, nr, 1);
        const uint16_t* lg = static_cast<const uint16_t*>(logits) + size_t(r0) * size_t(row_stride);
        int32_t* pk = pick + r0;
        uint8_t* fl = flag + r0;
        cudaError_t e = vec ? cudaLaunchKernelEx(&cfg, argmax_rows_kernel<true>, lg, V, row_stride, chunk, pk, fl)
                            : cudaLaunchKernelEx(&cfg, argmax_rows_kernel<false>, lg, V, row_stride, chunk, pk, fl);
        if (e != cudaSuccess) return cuda_fail(e);
        const int st = launch_status();
        if (st != TF_OK) return st;
    }
    return TF_OK;
}
