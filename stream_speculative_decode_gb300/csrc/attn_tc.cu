// a2 on the 5th-generation tensor cores: causal GQA attention partials with
// tcgen05 MMAs, accumulators in tensor memory and K/V tiles staged by TMA.
//
// Same work items, chunking and partial records as the mma.sync kernel in
// attn.cu (PR #1377 "LFM2: shared-round decode": one launch a layer over every
// row from the segment table, per-stream partials; PR #1391: causal count),
// used when a window holds 13 rows or more, where q.K and P.V are real
// contractions (4*rows flops per byte of K/V each) and the mma.sync kernel
// would need a fourth 16-row query tile. With `full` set it is the
// drafter's non-causal block attention (PR #1391: every block row sees the
// keys [0, len + 1)): only the per-row key bounds change.
//
// One CTA per (work item = one stream's key chunk, KV head), 7 warps:
//   warp 6, lane 0   TMA loads of K/V tiles (64 keys = 8 KB each, 128-byte
//                    swizzle) into a 5-stage ring, refilling a stage as soon
//                    as the P.V that read it completes;
//   warp 4, lane 0   the MMAs;
//   warp 5           converts each V tile bf16 -> fp16 in shared memory as
//                    soon as it lands (exact within fp16's range);
//   warps 0-3        softmax; query row qi sits on TMEM lane
//                    32*(qi / per) + qi % per (per = ceil(4*rows / 4)), so the
//                    rows spread over the four lane quadrants and all four
//                    SM sub-partitions share the softmax.
// Per key tile j (TMEM columns: S/P of tile j at 64*(j%3), O at 192):
//   S = Q K^T      M = 128 lanes (4*rows real rows, the rest zero), N = 64
//                  keys, K = 64: A = Q (bf16, smem), B = K tile (bf16, smem);
//                  issued while the softmax still works on tile j-1;
//   softmax        thread = query row: the 64 scores in registers (one TMEM
//                  load), row max, lazy rescale of O (only when the max rises
//                  more than 2^8), p = 2^(s*log2e/8 - m) packed to fp16 in
//                  place of S;
//   O += P V       A = P (fp16, tensor memory), B = V tile (fp16, smem,
//                  MN-major), fp32 accumulate.
// S/P has three buffers, so the q.K of tile j waits only for the P.V of
// tile j-3 and is ready before the softmax reaches it.
// At the end (m, l, O) is renormalised to the true running max and written
// as the chunk's partial records.
//
// Every wait on an mbarrier is bounded (2 s of %globaltimer); on a timeout the
// CTA raises a shared abort flag, waits (bounded) for its TMA copies and MMAs
// in flight, writes NaN records (so the merged output shows the failure),
// frees its tensor memory and returns.
#include "tc_ptx.cuh"

namespace tf {
namespace {

constexpr int kKT = 64;                     // keys per tile
constexpr int kStages = 5;
constexpr int kTileB = kKT * TF_D * 2;      // 8 KB: one K or V tile
constexpr int kStageB = 2 * kTileB;         // K then V
constexpr int kQRows = 128;                 // MMA M
constexpr int kQB = kQRows * TF_D * 2;      // 16 KB
constexpr int kWarps = 7;
constexpr int kThreads = kWarps * 32;
constexpr uint32_t kCols = 256;             // tensor-memory columns per CTA
constexpr int kSBuf = 3;                    // S/P buffers: tile j uses buffer j % 3
constexpr uint32_t kColS = 0;               // + 64 * (tile % 3)
constexpr uint32_t kColO = 192;             // O: 64 columns
constexpr float kLog2e8 = 0.18033688011112042f;   // log2(e) / sqrt(64)
constexpr float kTau = 8.f;

struct Bars {
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t v_ready[kStages];   // the stage's V tile is converted to fp16
    uint64_t s_full[kSBuf];      // per S buffer
    uint64_t p_full[kSBuf];      // per S buffer
    uint64_t o_done[kSBuf];      // P.V of a tile using S buffer b completed
    uint64_t drain;
    uint32_t tmem_base;
    uint32_t abort_flag;
};
constexpr int kSmemBytes = 1024 + kQB + kStages * kStageB + int(sizeof(Bars));

// Instruction descriptors, kind::f16, fp32 accumulate, M = 128, N = 64.
//   bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format (0 = f16, 1 = bf16),
//   15/16 A/B major (0 = K-major, 1 = MN-major), 17-22 N >> 3, 24-28 M >> 4.
constexpr uint32_t kIdescQK = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(64 >> 3) << 17) |
                              (uint32_t(128 >> 4) << 24);
constexpr uint32_t kIdescPV = (1u << 4) | (1u << 16) | (uint32_t(64 >> 3) << 17) | (uint32_t(128 >> 4) << 24);

__device__ __forceinline__ float ex2(float x) { return ex2_approx(x); }
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w) {
    return pack_h2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// State of one softmax thread: query row qi = per*(lane quadrant) + lane sits
// on TMEM lane quadrant*32 + lane (lanes past `per` hold zero rows).
struct SoftState {
    Bars* bars;
    volatile uint32_t* abortp;
    uint32_t trow;       // TMEM address of the warp's lane quadrant
    int T, lim, lim_all;
    bool wact;           // the warp holds at least one real query row
    float mref, mtrue;   // reference (lazy) and true running max, log2 units
    float l;             // sum of 2^(s*log2e/8 - mref) over the keys so far
};

template <int KC>
__device__ __forceinline__ void softmax_tiles(SoftState& st) {
    const int lane = threadIdx.x & 31;
    Bars* bars = st.bars;
    for (int j = 0; j < st.T; ++j) {
        const int b = j % kSBuf;
        const uint32_t colS = kColS + 64 * b;
        if (!mbar_wait(su32(&bars->s_full[b]), (j / kSBuf) & 1, st.abortp)) break;
        tc_fence_after();
        if (st.wact) {
            const int k0 = j * kKT;                  // chunk-local first key of the tile
            float v[KC];
            {
                uint32_t r[KC];
                tc_ld_n<KC>(st.trow + colS, r);
                tc_wait_ld();
#pragma unroll
                for (int c = 0; c < KC; ++c) v[c] = __uint_as_float(r[c]);
            }
            if (j * kKT + kKT > st.lim_all) {   // the causal edge or the chunk's end lies in this tile
#pragma unroll
                for (int c = 0; c < KC; ++c)
                    if (k0 + c >= st.lim) v[c] = -INFINITY;
            }
            float m8[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                m8[a] = v[a];
#pragma unroll
                for (int c = a + 8; c < KC; c += 8) m8[a] = fmaxf(m8[a], v[c]);
            }
            const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            const float mxs = mx * kLog2e8;
            st.mtrue = fmaxf(st.mtrue, mxs);
            const bool resc = mxs > st.mref + kTau;
            if (__any_sync(0xFFFFFFFFu, resc)) {
                // O holds P.V of tiles < j; the last of them (j-1) must be done
                if (j >= 1 && !mbar_wait(su32(&bars->o_done[(j - 1) % kSBuf]), ((j - 1) / kSBuf) & 1, st.abortp))
                    break;
                tc_fence_after();
                const float alpha = resc ? ex2(st.mref - mxs) : 1.f;
                if (resc) {
                    st.mref = mxs;
                    st.l *= alpha;
                }
                if (j >= 1) {
#pragma unroll 1
                    for (int h = 0; h < 4; ++h) {   // O (64 columns)
                        uint32_t o16[16];
                        tc_ld16(st.trow + kColO + 16 * h, o16);
                        tc_wait_ld();
                        uint32_t a8[8], b8[8];
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            a8[c] = __float_as_uint(__uint_as_float(o16[c]) * alpha);
                            b8[c] = __float_as_uint(__uint_as_float(o16[8 + c]) * alpha);
                        }
                        tc_st8(st.trow + kColO + 16 * h, a8);
                        tc_st8(st.trow + kColO + 16 * h + 8, b8);
                    }
                    tc_wait_st();
                }
            }
            const float mu = (st.mref == -INFINITY) ? 0.f : st.mref;
            uint32_t own[KC / 2];
            float s4[4] = {0.f, 0.f, 0.f, 0.f};   // four independent sums
#pragma unroll
            for (int c = 0; c < KC / 2; ++c) {
                const float p0 = ex2(fmaf(v[2 * c], kLog2e8, -mu));
                const float p1 = ex2(fmaf(v[2 * c + 1], kLog2e8, -mu));
                s4[c & 3] += p0 + p1;
                own[c] = pack_h2(p0, p1);
            }
            tc_st_n<KC / 2>(st.trow + colS, own);   // P (fp16 pairs) over the first KC/2 columns of S
            st.l += (s4[0] + s4[1]) + (s4[2] + s4[3]);
            tc_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(su32(&bars->p_full[b]));
    }
}

__global__ void __launch_bounds__(kThreads, 2)
attn_partials_tc_kernel(SegTable t, int layer, const uint16_t* __restrict__ q, float* __restrict__ part_o,
                        float2* __restrict__ part_ml, float* __restrict__ out, int full) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = su32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;            // 128-byte swizzle atoms need 1 KB alignment
    unsigned char* gbase = smem_raw + (base - raw);
    const uint32_t sQ = base;
    const uint32_t sStage = base + kQB;
    Bars* bars = reinterpret_cast<Bars*>(gbase + kQB + kStages * kStageB);
    volatile uint32_t* abortp = &bars->abort_flag;

    const int item_idx = t.n_items_mma + blockIdx.x / TF_NKV;   // tensor-core items follow the mma.sync ones
    const int g = blockIdx.x % TF_NKV;
    const AttnItem item = t.items[item_idx];
    const SegStream st = t.streams[item.stream];
    const int nq = st.rows * 4;
    const int mode = out ? st.merge_mode : kMergeKernel;   // records only in the two-call form
    // query rows per TMEM lane quadrant: rows spread over the four quadrants so
    // that all four SM sub-partitions share the softmax
    const int per = (nq + 3) / 4;
    const int c0 = item.chunk * st.chunk_keys;
    const int nkeys = min(st.chunk_keys, st.keys - c0);
    const int T = (nkeys + kKT - 1) / kKT;
    const size_t slot = size_t(layer) * t.S + item.stream;
    const CUtensorMap* kmap = t.k_maps + slot;
    const CUtensorMap* vmap = t.v_maps + slot;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(su32(&bars->kv_full[s]), 1);
            mbar_init(su32(&bars->kv_empty[s]), 1);
            mbar_init(su32(&bars->v_ready[s]), 1);
        }
        for (int b = 0; b < kSBuf; ++b) {
            mbar_init(su32(&bars->s_full[b]), 1);
            mbar_init(su32(&bars->p_full[b]), 4);   // the 4 softmax warps
            mbar_init(su32(&bars->o_done[b]), 1);
        }
        mbar_init(su32(&bars->drain), 1);
        bars->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_wait();   // the table above; queries and caches below
    if (warp == 4) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(su32(&bars->tmem_base)), "r"(kCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    } else if (warp < 4) {
        // Q rows on their lanes (zero elsewhere), swizzled K-major: lane L holds
        // query qi = per*(L/32) + L%32 when L%32 < per and qi < 4*rows
        for (int idx = tid; idx < kQRows * 8; idx += 128) {
            const int L = idx >> 3, ch = idx & 7;
            const int qq = per * (L >> 5) + (L & 31);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if ((L & 31) < per && qq < nq)
                v = *reinterpret_cast<const uint4*>(
                    q + ((size_t(st.row_offset + (qq >> 2)) * TF_NQ + 4 * g + (qq & 3)) * TF_D + ch * 8));
            sts128(sQ + L * 128 + ((ch ^ (L & 7)) << 4), v);
        }
        fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    // softmax-thread state (warps 0-3): this thread's TMEM lane, query row and key slice
    const int qi = per * warp + lane;
    const bool qvalid = warp < 4 && lane < per && qi < nq;
    const bool wact = warp < 4 && per * warp < nq;      // the warp holds at least one real row
    const uint32_t trow = tmem + (uint32_t(warp * 32) << 16);
    SoftState ss;
    ss.bars = bars;
    ss.abortp = abortp;
    ss.trow = trow;
    ss.T = T;
    // chunk-local key bounds: causal count of the row (of row 0 for lim_all),
    // or every key for a FULL block
    ss.lim = qvalid ? (full ? st.keys : st.keys - st.rows + (qi >> 2) + 1) - c0 : 0;
    ss.lim_all = (full ? st.keys : st.keys - st.rows + 1) - c0;
    ss.wact = wact;
    ss.mref = -INFINITY;
    ss.mtrue = -INFINITY;
    ss.l = 0.f;

    if (warp == 4) {
        // ------------------------------------------------------------ control
        if (lane == 0) {
            const uint64_t dq = sdesc(sQ, 16, 1024);
            bool ok = true;
            for (int j = 0; j <= T && ok; ++j) {
                if (j < T) {
                    const int s = j % kStages, b = j % kSBuf;
                    ok = mbar_wait(su32(&bars->kv_full[s]), (j / kStages) & 1, abortp);
                    if (!ok) break;
                    if (j >= kSBuf) {   // P.V(j-3) has released S buffer b
                        ok = mbar_wait(su32(&bars->o_done[b]), ((j - kSBuf) / kSBuf) & 1, abortp);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    const uint64_t dk = sdesc(sStage + s * kStageB, 16, 1024);
#pragma unroll
                    for (int k = 0; k < TF_D / 16; ++k)   // K = 64: 4 steps of 16 (32 bytes)
                        tc_mma_ss(tmem + kColS + 64 * b, dq + 2 * k, dk + 2 * k, kIdescQK, k > 0 ? 1u : 0u);
                    tc_commit(su32(&bars->s_full[b]));
                }
                if (j >= 1) {
                    const int jj = j - 1, s = jj % kStages, b = jj % kSBuf;
                    ok = mbar_wait(su32(&bars->p_full[b]), (jj / kSBuf) & 1, abortp);
                    if (!ok) break;
                    ok = mbar_wait(su32(&bars->v_ready[s]), (jj / kStages) & 1, abortp);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t dv = sdesc(sStage + s * kStageB + kTileB, kTileB, 1024);
#pragma unroll
                    for (int k = 0; k < kKT / 16; ++k)   // 64 keys: 4 steps of 16 (2 KB of V rows)
                        tc_mma_ts(tmem + kColO, tmem + kColS + 64 * b + 8 * k, dv + 128 * k, kIdescPV,
                                  (jj > 0 || k > 0) ? 1u : 0u);
                    tc_commit(su32(&bars->o_done[b]));
                    tc_commit(su32(&bars->kv_empty[s]));
                }
            }
            if (ok) mbar_wait(su32(&bars->kv_empty[(T - 1) % kStages]), ((T - 1) / kStages) & 1, abortp);
            tc_commit(su32(&bars->drain));   // every MMA issued so far
            mbar_drain(su32(&bars->drain), 0);
        }
        __syncwarp();
    } else if (warp == 6) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int j = 0; j < T; ++j) {
                const int s = j % kStages;
                if (j >= kStages &&   // the stage is free once the P.V of tile j - kStages completed
                    !mbar_wait(su32(&bars->kv_empty[s]), ((j - kStages) / kStages) & 1, abortp))
                    break;
                const uint32_t bar = su32(&bars->kv_full[s]);
                mbar_expect_tx(bar, kStageB);
                tma_load_3d(sStage + s * kStageB, kmap, 0, c0 + j * kKT, g, bar);
                tma_load_3d(sStage + s * kStageB + kTileB, vmap, 0, c0 + j * kKT, g, bar);
                ++issued;
            }
            if (*abortp)   // let the copies in flight land before the CTA exits
                for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
                    mbar_drain(su32(&bars->kv_full[j % kStages]), (j / kStages) & 1);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------------ softmax
        softmax_tiles<kKT>(ss);
        if (!*abortp) mbar_wait(su32(&bars->o_done[(T - 1) % kSBuf]), ((T - 1) / kSBuf) & 1, abortp);
    } else {
        // ------------------------------------------------------------ V tiles bf16 -> fp16
        for (int j = 0; j < T; ++j) {
            const int s = j % kStages;
            if (!mbar_wait(su32(&bars->kv_full[s]), (j / kStages) & 1, abortp)) break;
            const uint32_t vs = sStage + s * kStageB + kTileB;
#pragma unroll
            for (int c = 0; c < kTileB / 16 / 32; ++c) {
                const uint32_t a = vs + uint32_t(lane + 32 * c) * 16u;
                uint4 v = lds128(a);
                v.x = bf2_to_h2(v.x);
                v.y = bf2_to_h2(v.y);
                v.z = bf2_to_h2(v.z);
                v.w = bf2_to_h2(v.w);
                sts128(a, v);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(su32(&bars->v_ready[s]));
            // the stage is refilled only after this tile's P.V, which waits on
            // this arrival, so the next use of this stage cannot overtake it
        }
    }
    tc_fence_before();
    __syncthreads();   // every MMA and copy of the CTA is done
    tc_fence_after();
    pdl_trigger();

    if (wact) {
        // (m, l, O) renormalised to the true running max -> the chunk's record
        const bool aborted = *abortp != 0;
        float f = 1.f;
        if (ss.mtrue > ss.mref && ss.mref != -INFINITY) f = ex2(ss.mref - ss.mtrue);
        uint32_t ro[64];
        tc_ld64(trow + kColO, ro);
        tc_wait_ld();
        const float lsum = ss.l;
        float o[64];
#pragma unroll
        for (int d = 0; d < 64; ++d) o[d] = __uint_as_float(ro[d]);
        if (qvalid && mode == kMergeDirect) {   // the stream's only chunk: the output itself
            const float inv = aborted ? NAN : 1.f / lsum;   // a row always sees key 0 of its stream
            float4* dst = reinterpret_cast<float4*>(out_row(out, st, g, qi));
#pragma unroll
            for (int c = 0; c < 16; ++c)
                dst[c] = make_float4(o[4 * c] * inv, o[4 * c + 1] * inv, o[4 * c + 2] * inv, o[4 * c + 3] * inv);
        } else if (qvalid) {
            const int64_t rec = st.pbase + (int64_t(item.chunk) * TF_NKV + g) * nq + qi;
            const bool empty = ss.mtrue == -INFINITY;
            float4* dst = reinterpret_cast<float4*>(part_o + rec * TF_D);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                float4 v = make_float4(o[4 * c] * f, o[4 * c + 1] * f, o[4 * c + 2] * f, o[4 * c + 3] * f);
                if (aborted) v = make_float4(NAN, NAN, NAN, NAN);
                else if (empty) v = make_float4(0.f, 0.f, 0.f, 0.f);
                dst[c] = v;
            }
            part_ml[rec] = aborted ? make_float2(NAN, INFINITY)
                                   : make_float2(ss.mtrue, empty ? 0.f : lsum * f);
        }
    }
    if (mode == kMergeLastCta) {
        __shared__ int last_flag;
        finish_last_cta(t, layer, item.stream, st, g, part_o, part_ml, out, &last_flag);
    }
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
    }
}

}  // namespace

int attn_tc_prepare() {
    cudaError_t e = cudaFuncSetAttribute(attn_partials_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    return e == cudaSuccess ? TF_OK : cuda_fail(e);
}

int launch_attn_partials_tc(const SegTable& t, int layer, const uint16_t* q, float* po, float2* pml,
                            cudaStream_t stream, float* out, int full) {
    if (!t.k_maps || !t.v_maps) return TF_EINVAL;
    return launch_pdl(attn_partials_tc_kernel, dim3((t.n_items - t.n_items_mma) * TF_NKV), dim3(kThreads),
                      kSmemBytes, stream, t, layer, q, po, pml, out, full);
}

}  // namespace tf
