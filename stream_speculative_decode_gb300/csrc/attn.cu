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
// cache; a wider one reads it once per group, the later groups from L2. Four
// warps split each stage's keys (16 each); every warp keeps an online softmax
// over its keys for all query rows; the warps are combined at the end. q.k runs on bf16 tensor-core MMAs with fp32 accumulation (exact
// products); P.V runs with P and V in fp16 (V's bf16 values convert exactly
// within fp16's range) and fp32 accumulation.
//
// HBM bound: 256 bytes of K+V per key per KV head; the window's queries ride
// along. Arithmetic intensity 4*rows flops per byte for each of q.k and P.V.
//
// The same kernels serve the drafter's block attention (PR #1391: the target's
// attention and merge "with a FULL template flag", every block row seeing the
// keys [0, len + 1)): with `full` set every window row sees all of the
// stream's keys instead of its causal count; nothing else changes, and the
// merge is shared (it reads only the records).
#include "tf_internal.cuh"

namespace tf {
namespace {

constexpr int kKT = 64;                 // keys per stage
constexpr int kStages = 4;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRowB = TF_D * 2;         // 128 bytes per cache row
constexpr int kStageB = 2 * kKT * kRowB;  // K then V: 16 KB
constexpr int kOStride = 68;            // floats per row of the warp-combine buffer
constexpr float kLog2e8 = 0.18033688011112042f;   // log2(e) / sqrt(64)
constexpr float kTau = 8.f;             // lazy-rescale threshold, log2 units

__host__ __device__ constexpr int smem_bytes(int mt) { return kStages * kStageB + 16 * mt * kRowB; }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    const int sz = valid ? 16 : 0;   // 0: fill the 16 bytes with zeros
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t r[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t r[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
// two bf16 -> two fp16 (exact for |v| in fp16's normal range)
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w) {
    return pack_h2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
// byte offset of 16-byte chunk `ch` of row `r` in a swizzled 128-byte-row tile
__device__ __forceinline__ uint32_t swz(int r, int ch) { return uint32_t(r * kRowB + ((ch ^ (r & 7)) << 4)); }

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
    constexpr bool kQReg = MT <= 2;
    const int item_idx = blockIdx.x / TF_NKV;
    const int g = blockIdx.x % TF_NKV;
    const AttnItem item = t.items[item_idx];
    const SegStream st = t.streams[item.stream];
    const int nq_all = st.rows * 4;
    const int q0 = item.q0;                   // the group's first query row (a multiple of 32)
    const int nq = min(16 * MT, nq_all - q0);   // the group's query rows
    const int c0 = item.chunk * st.chunk_keys;
    const int nkeys = min(st.chunk_keys, st.keys - c0);
    const int nst = (nkeys + kKT - 1) / kKT;
    const size_t slot = size_t(layer) * t.S + item.stream;
    const uint16_t* Kg = static_cast<const uint16_t*>(t.k_cache[slot]) + (size_t(g) * st.cap + c0) * TF_D;
    const uint16_t* Vg = static_cast<const uint16_t*>(t.v_cache[slot]) + (size_t(g) * st.cap + c0) * TF_D;
    unsigned char* sKV = smem;
    unsigned char* sQ = smem + kStages * kStageB;
    const uint32_t sKV32 = smem_u32(sKV), sQ32 = smem_u32(sQ);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if constexpr (MT == 1) {
        // narrow windows (one m-tile: short launches, one wave): the first
        // stages' keys and values into L2 while the previous kernel finishes
        // (measured 17.0 -> 16.0 us a layer for 16 one-row streams; the
        // two-m-tile kernel spilled with it and ran slower)
        if (tid == 0) {
            const uint32_t pre = uint32_t(min(nkeys, (kStages - 1) * kKT)) * kRowB;
            l2_prefetch_bulk(Kg, pre);
            l2_prefetch_bulk(Vg, pre);
        }
    }
    pdl_wait();   // the table above; queries and caches below

    // group query rows qi: q0 + qi = 4*i + hh (window row i, head 4g + hh);
    // rows past nq are zero
    for (int idx = tid; idx < 16 * MT * 8; idx += kThreads) {
        const int qi = idx >> 3, ch = idx & 7;
        const bool valid = qi < nq;
        const uint16_t* src =
            q + ((size_t(st.row_offset + ((q0 + qi) >> 2)) * TF_NQ + 4 * g + (qi & 3)) * TF_D + ch * 8);
        cp_async16(sQ32 + swz(qi, ch), valid ? src : q, valid);
    }
    auto issue = [&](int s) {
        const uint32_t buf = sKV32 + (s % kStages) * kStageB;
        const int key0 = s * kKT;
#pragma unroll
        for (int k = 0; k < (kKT * 8) / kThreads; ++k) {
            const int idx = tid + k * kThreads;
            const int r = idx >> 3, ch = idx & 7;
            const bool valid = key0 + r < nkeys;
            const size_t off = size_t(key0 + r) * TF_D + ch * 8;
            cp_async16(buf + swz(r, ch), valid ? Kg + off : Kg, valid);
            cp_async16(buf + kKT * kRowB + swz(r, ch), valid ? Vg + off : Vg, valid);
        }
    };
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < nst) issue(s);
        cp_async_commit();
    }

    const int g8 = lane >> 2, t4 = lane & 3;
    float o[MT][8][4];
    float m[MT][2], l[MT][2], mtrue[MT][2];   // m: reference max; mtrue: running max
    int lim[MT][2];
    // keys every real row of the group sees (chunk-local): its first row's
    // causal count, or every key for a FULL block
    const int lim_all = (full ? st.keys : st.keys - st.rows + (q0 >> 2) + 1) - c0;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int dt = 0; dt < 8; ++dt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[mt][dt][e] = 0.f;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            m[mt][r] = -INFINITY;
            mtrue[mt][r] = -INFINITY;
            l[mt][r] = 0.f;
            const int qi = mt * 16 + g8 + 8 * r;
            // chunk-local bound of the keys row qi/4 sees (causal, or all keys
            // for a FULL block), 0 for padding rows
            const int vis = (full ? st.keys : st.keys - st.rows + ((q0 + qi) >> 2) + 1) - c0;
            lim[mt][r] = qi < nq ? max(0, min(vis, nkeys)) : 0;
        }
    }
    uint32_t qf[kQReg ? MT : 1][4][4];

    for (int it = 0; it < nst; ++it) {
        if (it + kStages - 1 < nst) issue(it + kStages - 1);
        cp_async_commit();
        cp_async_wait<kStages - 1>();
        __syncthreads();
        if (kQReg && it == 0) {
#pragma unroll
            for (int mt = 0; mt < (kQReg ? MT : 0); ++mt)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const int mi = lane >> 3;
                    const int row = mt * 16 + (mi & 1) * 8 + (lane & 7);
                    ldsm_x4(qf[mt][ks], sQ32 + swz(row, ks * 2 + (mi >> 1)));
                }
        }
        const int kw0 = it * kKT + warp * 16;   // chunk-local first key of this warp
        if (kw0 < nkeys) {
            const uint32_t bufK = sKV32 + (it % kStages) * kStageB;
            const uint32_t bufV = bufK + kKT * kRowB;
            uint32_t kb[4][4];
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const int mi = lane >> 3;
                const int r = warp * 16 + (mi >> 1) * 8 + (lane & 7);
                ldsm_x4(kb[ks], bufK + swz(r, ks * 2 + (mi & 1)));
            }
            uint32_t vb[8][2];
#pragma unroll
            for (int dp = 0; dp < 4; ++dp) {
                const int mi = lane >> 3;
                const int r = warp * 16 + (mi & 1) * 8 + (lane & 7);
                uint32_t x[4];
                ldsm_x4_t(x, bufV + swz(r, dp * 2 + (mi >> 1)));
                vb[2 * dp][0] = bf2_to_h2(x[0]);
                vb[2 * dp][1] = bf2_to_h2(x[1]);
                vb[2 * dp + 1][0] = bf2_to_h2(x[2]);
                vb[2 * dp + 1][1] = bf2_to_h2(x[3]);
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                if (mt * 16 < nq) {
                    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        uint32_t a[4];
                        if (kQReg) {
#pragma unroll
                            for (int k = 0; k < 4; ++k) a[k] = qf[kQReg ? mt : 0][ks][k];
                        } else {
                            const int mi = lane >> 3;
                            const int row = mt * 16 + (mi & 1) * 8 + (lane & 7);
                            ldsm_x4(a, sQ32 + swz(row, ks * 2 + (mi >> 1)));
                        }
                        mma_bf16(s[0], a, kb[ks][0], kb[ks][1]);
                        mma_bf16(s[1], a, kb[ks][2], kb[ks][3]);
                    }
                    // scores of row 0 and every later row are all visible up to
                    // lim_all; past it (the causal edge, the chunk's end) mask
                    if (kw0 + 16 > lim_all) {
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int key = kw0 + nt * 8 + 2 * t4 + (e & 1);
                                if (key >= lim[mt][e >> 1]) s[nt][e] = -INFINITY;
                            }
                    }
                    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) mx[e >> 1] = fmaxf(mx[e >> 1], s[nt][e]);
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xFFFFFFFFu, mx[r], 1));
                        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xFFFFFFFFu, mx[r], 2));
                    }
                    // lazy rescale: the reference max moves only when a row's max
                    // rises more than kTau (log2 units) above it, so p <= 2^kTau
                    float alpha[2] = {1.f, 1.f}, muse[2];
                    bool resc = false;
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const float mxs = mx[r] * kLog2e8;
                        mtrue[mt][r] = fmaxf(mtrue[mt][r], mxs);
                        if (mxs > m[mt][r] + kTau) {
                            alpha[r] = ex2(m[mt][r] - mxs);
                            m[mt][r] = mxs;
                            resc = true;
                        }
                        muse[r] = (m[mt][r] == -INFINITY) ? 0.f : m[mt][r];
                    }
                    if (__any_sync(0xFFFFFFFFu, resc)) {
#pragma unroll
                        for (int r = 0; r < 2; ++r) l[mt][r] *= alpha[r];
#pragma unroll
                        for (int dt = 0; dt < 8; ++dt) {
                            o[mt][dt][0] *= alpha[0];
                            o[mt][dt][1] *= alpha[0];
                            o[mt][dt][2] *= alpha[1];
                            o[mt][dt][3] *= alpha[1];
                        }
                    }
                    float ps[2] = {0.f, 0.f};
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float p = ex2(fmaf(s[nt][e], kLog2e8, -muse[e >> 1]));
                            s[nt][e] = p;
                            ps[e >> 1] += p;
                        }
#pragma unroll
                    for (int r = 0; r < 2; ++r) l[mt][r] += ps[r];
                    uint32_t pa[4];
                    pa[0] = pack_h2(s[0][0], s[0][1]);
                    pa[1] = pack_h2(s[0][2], s[0][3]);
                    pa[2] = pack_h2(s[1][0], s[1][1]);
                    pa[3] = pack_h2(s[1][2], s[1][3]);
#pragma unroll
                    for (int dt = 0; dt < 8; ++dt) mma_f16(o[mt][dt], pa, vb[dt][0], vb[dt][1]);
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();
    __syncthreads();
    pdl_trigger();

    // renormalise each row to its true running max (exact partial format)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            if (mtrue[mt][r] > m[mt][r]) {
                const float f = ex2(m[mt][r] - mtrue[mt][r]);
                l[mt][r] *= f;
#pragma unroll
                for (int dt = 0; dt < 8; ++dt) {
                    o[mt][dt][2 * r] *= f;
                    o[mt][dt][2 * r + 1] *= f;
                }
            }
            m[mt][r] = mtrue[mt][r];
        }

    // ---- combine the four warps (shared memory reused)
    float* sO = reinterpret_cast<float*>(smem);                     // [4][16*MT][kOStride]
    float* sM = sO + kWarps * 16 * MT * kOStride;                    // [4][16*MT]
    float* sL = sM + kWarps * 16 * MT;                               // [4][16*MT]
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float lr = l[mt][r];
            lr += __shfl_xor_sync(0xFFFFFFFFu, lr, 1);
            lr += __shfl_xor_sync(0xFFFFFFFFu, lr, 2);
            const int qi = mt * 16 + g8 + 8 * r;
            if (t4 == 0) {
                sM[warp * 16 * MT + qi] = m[mt][r];
                sL[warp * 16 * MT + qi] = lr;
            }
            float* row = sO + (size_t(warp) * 16 * MT + qi) * kOStride;
#pragma unroll
            for (int dt = 0; dt < 8; ++dt)
                *reinterpret_cast<float2*>(row + dt * 8 + 2 * t4) =
                    make_float2(o[mt][dt][2 * r], o[mt][dt][2 * r + 1]);
        }
    }
    __syncthreads();
    const int mode = out ? st.merge_mode : kMergeKernel;   // records only in the two-call form
    const int64_t rec0 = st.pbase + (int64_t(item.chunk) * TF_NKV + g) * nq_all + q0;
    for (int idx = tid; idx < nq * (TF_D / 4); idx += kThreads) {
        const int qi = idx >> 4, d4 = (idx & 15) * 4;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sM[w * 16 * MT + qi]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float L = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float mw = sM[w * 16 * MT + qi];
                const float wt = (mw == -INFINITY) ? 0.f : ex2(mw - M);
                L += wt * sL[w * 16 * MT + qi];
                const float4 v = *reinterpret_cast<const float4*>(sO + (size_t(w) * 16 * MT + qi) * kOStride + d4);
                acc.x += wt * v.x;
                acc.y += wt * v.y;
                acc.z += wt * v.z;
                acc.w += wt * v.w;
            }
        }
        if (mode == kMergeDirect) {   // the stream's only chunk: the output itself
            const float inv = 1.f / L;
            *reinterpret_cast<float4*>(out_row(out, st, g, q0 + qi) + d4) =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        } else {
            *reinterpret_cast<float4*>(part_o + (rec0 + qi) * TF_D + d4) = acc;
            if (d4 == 0) part_ml[rec0 + qi] = make_float2(M, L);
        }
    }
    if (mode == kMergeLastCta) {
        __shared__ int last_flag;
        finish_last_cta<MT == 1 ? 8 : 16>(t, layer, item.stream, st, g, part_o, part_ml, out, &last_flag);
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
