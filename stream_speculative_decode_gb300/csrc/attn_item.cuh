// The mma.sync attention of one work item: one key chunk of one stream, one
// KV head, at most 2 x 16 query rows (at most 8 window rows times their 4
// query heads), by 128 threads (4 warps) of a CTA. Shared by the mma.sync
// partials kernel (attn.cu), which runs one item per CTA, and the tensor-core
// kernel (attn_tc.cu), whose last CTA recomputes with it the rare units that
// need P.V exact in V.
//
// PR #1377 "LFM2: shared-round decode": commit "the conv, qk, attention and
// merge kernels' bodies as inline functions" (qk, attention, merge) and commit
// "a shared round runs each layer's conv and attention once over all its
// streams" (per-stream partials); PR #1391: the target's attention keeps its
// causal count, and the FULL (block) form sees every key.
//
// Four warps split each 64-key stage (16 keys each); every warp keeps an
// online softmax over its keys for all query rows; the warps are combined at
// the end. q.k runs on bf16 tensor-core MMAs with fp32 accumulation (exact
// products). P.V: see attn_item.
#pragma once

#include <type_traits>

#include "tf_internal.cuh"

namespace tf {
namespace item {

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
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void mma_f16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
// two bf16 -> two fp16 (exact for |v| in fp16's normal range)
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w) {
    return pack_h2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
// Two fp32 probabilities (a low, b high) as bf16 pairs: hi = their top 16
// bits (bf16 rounded toward zero), lo = the remainders a - hi_a, b - hi_b
// (exact in fp32) rounded to nearest bf16. hi + lo is a and b to about 2^-16
// relative.
__device__ __forceinline__ void split_bf2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
    hi = __byte_perm(ua, ub, 0x7632);
    __nv_bfloat162 r = __floats2bfloat162_rn(a - __uint_as_float(ua & 0xFFFF0000u),
                                             b - __uint_as_float(ub & 0xFFFF0000u));
    lo = *reinterpret_cast<uint32_t*>(&r);
}
// byte offset of 16-byte chunk `ch` of row `r` in a swizzled 128-byte-row tile
__device__ __forceinline__ uint32_t swz(int r, int ch) { return uint32_t(r * kRowB + ((ch ^ (r & 7)) << 4)); }

// Barrier `id` of the item's 128 threads (id 0 is the whole CTA of a 128-thread
// kernel), plain and with an OR / AND of a predicate over the 128 threads.
__device__ __forceinline__ void bar_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }
__device__ __forceinline__ bool bar_or(int id, bool x) {
    uint32_t r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, %2, 128, q;\n selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(r) : "r"(uint32_t(x)), "r"(id) : "memory");
    return r != 0;
}
__device__ __forceinline__ bool bar_and(int id, bool x) {
    uint32_t r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, %2, 128, q;\n selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(r) : "r"(uint32_t(x)), "r"(id) : "memory");
    return r != 0;
}

// Attention partials of one work item (stream item.stream, whose table row is
// st; key chunk item.chunk; query rows [item.q0, item.q0 + 32) of KV head g)
// by the 128 threads tid = 0..127, which meet at named barrier kBar, with
// `smem` (128-byte aligned, smem_bytes(MT)):
//   mode kMergeDirect writes the rows' output to `out`, any other mode the
//   chunk's partial records (m, l, o) to part_o / part_ml;
//   kFast: pass 0 runs P.V with P and V in fp16 (fp32 accumulation); pass 1,
//   taken only when pass 0 left a partial sum that is not finite (a V of
//   65,536 or more has no fp16 value) or every row's partial output below
//   2^-10 (V so small that fp16's subnormal steps of 2^-24 would cost
//   relative precision), recomputes the item with V in bf16 and P split into
//   a bf16 high part (its top 16 bits) and the bf16 rounding of the
//   remainder, two bf16 MMAs accumulating both: exact in V, P to about
//   2^-16. Without kFast only pass 1 runs. In a pass-0 result only values of
//   V below 2^-14 round, by at most 2^-25 each.
//   trigger: let the stream's next kernel launch once the passes are done.
// The caller has passed griddepcontrol.wait.
template <int MT, bool kFast, int kBar>
__device__ __forceinline__ void attn_item(const SegTable& t, int layer, const AttnItem item, const SegStream& st,
                                          int g, const uint16_t* __restrict__ q, float* __restrict__ part_o,
                                          float2* __restrict__ part_ml, float* __restrict__ out, int mode, int full,
                                          unsigned char* smem, int tid, bool trigger) {
    constexpr bool kQReg = MT <= 2;
    constexpr int bar = kBar;
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
    const int warp = tid >> 5, lane = tid & 31;

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
    const int g8 = lane >> 2, t4 = lane & 3;
    float o[MT][8][4];
    float m[MT][2], l[MT][2], mtrue[MT][2];   // m: reference max; mtrue: running max
    int lim[MT][2];
    // keys every real row of the group sees (chunk-local): its first row's
    // causal count, or every key for a FULL block
    const int lim_all = (full ? st.keys : st.keys - st.rows + (q0 >> 2) + 1) - c0;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int qi = mt * 16 + g8 + 8 * r;
            // chunk-local bound of the keys row qi/4 sees (causal, or all keys
            // for a FULL block), 0 for padding rows
            const int vis = (full ? st.keys : st.keys - st.rows + ((q0 + qi) >> 2) + 1) - c0;
            lim[mt][r] = qi < nq ? max(0, min(vis, nkeys)) : 0;
        }
    uint32_t qf[kQReg ? MT : 1][4][4];

    // Pass 0 runs P.V with V in fp16. Pass 1, taken only when pass 0 left a
    // partial sum that is not finite (a V of 65,536 or more became infinite
    // in fp16) or every row's partial output below 2^-10 (V so small that
    // fp16's subnormal steps would cost relative precision), recomputes the
    // item with V in bf16 and P split into two bf16 parts: exact in V.
    auto run_pass = [&](auto exact_tag) {
    constexpr bool vexact = decltype(exact_tag)::value;
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < nst) issue(s);
        cp_async_commit();
    }
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
        }
    }

    for (int it = 0; it < nst; ++it) {
        if (it + kStages - 1 < nst) issue(it + kStages - 1);
        cp_async_commit();
        cp_async_wait<kStages - 1>();
        bar_sync(bar);
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
                vb[2 * dp][0] = x[0];
                vb[2 * dp][1] = x[1];
                vb[2 * dp + 1][0] = x[2];
                vb[2 * dp + 1][1] = x[3];
            }
            if constexpr (!vexact) {   // V in fp16 (pass 0)
#pragma unroll
                for (int dt = 0; dt < 8; ++dt) {
                    vb[dt][0] = bf2_to_h2(vb[dt][0]);
                    vb[dt][1] = bf2_to_h2(vb[dt][1]);
                }
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
                    if constexpr (!vexact) {
                        uint32_t pa[4];
                        pa[0] = pack_h2(s[0][0], s[0][1]);
                        pa[1] = pack_h2(s[0][2], s[0][3]);
                        pa[2] = pack_h2(s[1][0], s[1][1]);
                        pa[3] = pack_h2(s[1][2], s[1][3]);
#pragma unroll
                        for (int dt = 0; dt < 8; ++dt) mma_f16(o[mt][dt], pa, vb[dt][0], vb[dt][1]);
                    } else {
                        uint32_t ph[4], pl[4];   // P as bf16 high parts and remainders
                        split_bf2(s[0][0], s[0][1], ph[0], pl[0]);
                        split_bf2(s[0][2], s[0][3], ph[1], pl[1]);
                        split_bf2(s[1][0], s[1][1], ph[2], pl[2]);
                        split_bf2(s[1][2], s[1][3], ph[3], pl[3]);
#pragma unroll
                        for (int dt = 0; dt < 8; ++dt) mma_bf16(o[mt][dt], ph, vb[dt][0], vb[dt][1]);
#pragma unroll
                        for (int dt = 0; dt < 8; ++dt) mma_bf16(o[mt][dt], pl, vb[dt][0], vb[dt][1]);
                    }
                }
            }
        }
        bar_sync(bar);
    }
    cp_async_wait<0>();
    bar_sync(bar);

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
    };
    if constexpr (kFast) {
    run_pass(std::false_type{});
    // whether pass 0 stands: every partial finite, and some row's |o| / l at
    // least 2^-10 (then fp16's subnormal steps, an absolute error of at most
    // 2^-25 per value, stay below 2^-15 of the largest output)
    bool nonfinite = false, tiny = true;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const float lr = l[mt][r];
            nonfinite |= !isfinite(lr);
#pragma unroll
            for (int dt = 0; dt < 8; ++dt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float v = o[mt][dt][2 * r + e];
                    nonfinite |= !isfinite(v);
                    tiny &= !(lr > 0.f && fabsf(v) >= 0x1p-10f * lr);   // rows without a key: no say
                }
        }
    if (bar_or(bar, nonfinite) | bar_and(bar, tiny)) run_pass(std::true_type{});
    } else {
        run_pass(std::true_type{});
    }
    if (trigger) pdl_trigger();

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
    bar_sync(bar);
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
}

}  // namespace item
}  // namespace tf
