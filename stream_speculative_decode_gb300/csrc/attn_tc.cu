// a2 on the 5th-generation tensor cores: causal GQA attention partials with
// tcgen05 MMAs, accumulators in tensor memory and K/V tiles staged by TMA.
//
// Same work items, chunking and partial records as the mma.sync kernel in
// attn.cu (PR #1377 "LFM2: shared-round decode": one launch a layer over every
// row from the segment table, per-stream partials; PR #1391: causal count),
// used when a window holds 9 rows or more, where q.K and P.V are real
// contractions (4*rows flops per byte of K/V each) and this kernel measured
// faster than the mma.sync one (which would take such a window as two items
// of at most 8 rows reading the chunk twice). With `full` set it is the
// drafter's non-causal block attention (PR #1391: all rows of a block share
// one key range, the stream's whole cache): only the per-row key bounds change.
//
// Persistent (at most two CTAs per SM, each running (key chunk, KV head)
// units back to back; see the kernel), 8 warps:
//   warp 6, lane 0   TMA loads of K/V tiles (64 keys = 8 KB each, 128-byte
//                    swizzle) into a 5-stage ring, refilling a stage as soon
//                    as the P.V that read it completes;
//   warp 4, lane 0   the q.K MMAs;
//   warp 7, lane 0   the P.V MMAs (two issuing threads: a single thread
//                    issuing both in tile order held each q.K behind the
//                    P.V of two tiles earlier, and the softmax waited for
//                    its scores);
//   warp 5           converts each V tile bf16 -> fp16 in shared memory as
//                    soon as it lands (exact within fp16's range); the
//                    second CTA on an SM swaps warps 5 and 6, so the two
//                    converters load different SM sub-partitions (the four
//                    softmax warps move in lockstep: the sub-partition with
//                    both converters set their pace);
//   warps 0-3        softmax; query row qi sits on TMEM lane
//                    32*(qi / per) + qi % per (per = 16 for windows of at
//                    most 16 rows, 32 for wider ones), so the rows spread
//                    over the four lane quadrants and all four SM
//                    sub-partitions share the softmax.
// The q.K thread also loads each unit's queries (TMA, 16 KB) as soon as the
// previous unit's last q.K has read the query buffer.
// Per key tile j (TMEM columns: S/P of tile j at 64*(j%3), O at 192):
//   S = Q K^T      M = 128 lanes (4*rows real rows, the rest zero), N = 64
//                  keys, K = 64: A = Q (bf16, smem), B = K tile (bf16, smem);
//                  issued while the softmax still works on tile j-1;
//   softmax        thread = query row: the 64 scores in registers (one TMEM
//                  load), p = 2^(s*log2e/8 - m) against the row's reference
//                  m, packed to fp16 in place of S; the tile's max only when
//                  the tile's sum of p passes 2^8 (it bounds every p) or the
//                  row has no reference yet, then a lazy rescale of O to the
//                  new reference; windows of at most 16 rows run it dual (two
//                  lanes per query row, 32 keys each, the row's two O
//                  halves added at the end);
//   O += P V       A = P (fp16, tensor memory), B = V tile (fp16, smem,
//                  MN-major), fp32 accumulate.
// S/P has three buffers, so the q.K of tile j waits only for the P.V of
// tile j-3 and is ready before the softmax reaches it.
// At the end (m, l, O) is renormalised to the true running max and written
// as the chunk's partial records.
//
// Every wait on an mbarrier is bounded (the library's wait limit, 2 s of
// %globaltimer unless tf_set_wait_limit_ns changed it); on a timeout the CTA
// raises a shared abort flag, waits (bounded) for its TMA copies and MMAs in
// flight, writes NaN records, sets TF_STATUS_ATTN_TIMEOUT in the table's
// status word, frees its tensor memory and returns.
#include "tc_ptx.cuh"
#include "attn_item.cuh"

namespace tf {
namespace {

// Launches per SM so far, by SM id: the second of two CTAs on an SM puts its
// V converter on another SM sub-partition than the first's (a load balance
// only: any outcome is correct).
__device__ unsigned int g_tc_sm_launches[1024];

constexpr int kKT = 64;                     // keys per tile
constexpr int kStages = 5;
constexpr int kTileB = kKT * TF_D * 2;      // 8 KB: one K or V tile
constexpr int kStageB = 2 * kTileB;         // K then V
constexpr int kQRows = 128;                 // MMA M
constexpr int kQB = kQRows * TF_D * 2;      // 16 KB
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr uint32_t kCols = 256;             // tensor-memory columns per CTA
constexpr int kSBuf = 3;                    // S/P buffers: tile j uses buffer j % 3
constexpr uint32_t kColS = 0;               // + 64 * (tile % 3)
constexpr uint32_t kColO = 192;             // O: 64 columns
constexpr float kLog2e8 = 0.18033688011112042f;   // log2(e) / sqrt(64)
constexpr float kSumMax = 256.f;            // 2^8: a tile whose p sum within it keeps its reference

constexpr int kUQ = 4;                      // queue of the CTA's next units
constexpr int kUQConsumers = 7;             // the two MMA threads, V converter warp, 4 softmax warps

struct Bars {
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t v_ready[kStages];   // the stage's V tile is converted to fp16
    uint64_t s_full[kSBuf];      // per S buffer
    uint64_t p_full[kSBuf];      // per S buffer
    uint64_t o_done[kSBuf];      // P.V of a tile using S buffer b completed
    uint64_t q_ready;            // the unit's queries are in shared memory (one phase a unit)
    uint64_t q_free;             // every q.K of the unit is done: its query buffer may be refilled
    uint64_t uq_full[kUQ];       // the CTA's next units (unit index, -1 when there are no more)
    uint64_t uq_empty[kUQ];
    int32_t uq[kUQ];
    uint64_t grp;                // the four softmax warps meet here (last-CTA merges)
    uint64_t drain;              // the q.K thread's MMAs in flight (drained at the end)
    uint64_t drain_pv;           // the P.V thread's
    uint32_t tmem_base;
    WaitCtl wc;                  // abort flag and wait limit of the CTA's bounded waits
    int32_t redo_m;              // the CTA's last unit (running index) queued for the exact recompute
    int32_t is_last;             // this CTA finished last (it runs the exact recomputes)
    int32_t last;
    int32_t alt;                 // this CTA swaps the producer and V-converter warps
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

// One unit of work: one key chunk of one stream (an attention item) for one
// KV head. A CTA takes the units blockIdx.x, blockIdx.x + gridDim.x, ... of the
// tensor-core items (largest first); every role walks the same list.
struct Unit {
    SegStream st;
    const CUtensorMap* kmap;
    const CUtensorMap* vmap;
    int stream, chunk, g, c0, T;
};
__device__ __forceinline__ Unit unit_of(const SegTable& t, int layer, int u) {
    Unit U;
    const AttnItem it = t.items[t.n_items_mma + u / TF_NKV];   // tensor-core items follow the mma.sync ones
    U.g = u % TF_NKV;
    U.stream = it.stream;
    U.chunk = it.chunk;
    U.st = t.streams[it.stream];
    U.c0 = it.chunk * U.st.chunk_keys;
    U.T = (min(U.st.chunk_keys, U.st.keys - U.c0) + kKT - 1) / kKT;
    const size_t slot = size_t(layer) * t.S + it.stream;
    U.kmap = t.k_maps + slot;
    U.vmap = t.v_maps + slot;
    return U;
}

// Blackwell's three-input max and paired fp32 FMA / add: each of these does
// the work of two instructions with the same per-element rounding.
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// p = 2^(s*log2e/8 - mu) for a thread's NV scores, two at a time, packed to
// fp16 pairs; returns the fp32 sum (two independent pair sums, added as
// ((s0 + s1) + (s2 + s3))). mu = 0 stands for a reference of -inf.
template <int NV>
__device__ __forceinline__ float exp_tile(const float (&v)[NV], float mref, uint32_t (&own)[NV / 2]) {
    const float mu = (mref == -INFINITY) ? 0.f : mref;
    const uint64_t k2 = f2pack(kLog2e8, kLog2e8), nmu2 = f2pack(-mu, -mu);
    uint64_t sum2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
#pragma unroll
    for (int c = 0; c < NV / 2; ++c) {
        float x0, x1;
        f2unpack(ffma2(f2pack(v[2 * c], v[2 * c + 1]), k2, nmu2), x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        sum2[c & 1] = fadd2(sum2[c & 1], f2pack(p0, p1));
        own[c] = pack_h2(p0, p1);
    }
    float s4[4];
    f2unpack(sum2[0], s4[0], s4[1]);
    f2unpack(sum2[1], s4[2], s4[3]);
    return (s4[0] + s4[1]) + (s4[2] + s4[3]);
}

// State of one softmax thread for one unit: query row qi = per*(lane quadrant)
// + lane sits on TMEM lane quadrant*32 + lane (lanes past `per` hold zero
// rows). Windows of at most 16 rows (per <= 16) run dual: lanes L and L + 16
// of a quadrant hold the same query, lane L scoring keys 0-31 of each tile
// and lane L + 16 keys 32-63, so every lane does useful softmax work.
struct SoftState {
    Bars* bars;
    volatile WaitCtl* abortp;
    uint32_t trow;       // TMEM address of the warp's lane quadrant
    int g0;              // the CTA's running tile count at the unit's first tile
    int T, lim, lim_all;
    bool wact;           // the warp holds at least one real query row
    float mref;          // reference max (lazy), log2 units: -inf until a tile gives the row a finite score
    float l;             // sum of 2^(s*log2e/8 - mref) over the keys so far
};

// DUAL (windows of at most 16 rows: the query rows sit on lanes 0-15 of each
// quadrant): threads L and L + 16 of a warp share TMEM lane L (the 16x32bx2
// load and store shape), thread L owning keys 0-31 of each tile and columns
// 0-31 of O, thread L + 16 keys 32-63 and columns 32-63; the row's max and sum
// are shared through one shuffle. Otherwise a thread owns its lane's row.
template <int KC, bool DUAL>
__device__ __forceinline__ void softmax_tiles(SoftState& st) {
    const int lane = threadIdx.x & 31;
    const int half = DUAL ? (lane >> 4) : 0;
    constexpr int NV = DUAL ? KC / 2 : KC;   // scores this thread owns per tile
    Bars* bars = st.bars;
    for (int j = 0; j < st.T; ++j) {
        const int gj = st.g0 + j;
        const int b = gj % kSBuf;
        const uint32_t colS = kColS + 64 * b;
        if (!mbar_wait_warp(su32(&bars->s_full[b]), (gj / kSBuf) & 1, st.abortp)) break;
        tc_fence_after();
        if (st.wact) {
            const int k0 = j * kKT + half * NV;      // chunk-local key of v[0]
            // this thread's scores of the tile, -inf past the row's last key
            auto load_scores = [&](float (&v)[NV]) {
                uint32_t r[NV];
                if constexpr (DUAL)
                    tc_ld16x2_32<KC / 2>(st.trow + colS, r);   // this half's 32 scores of lane L
                else
                    tc_ld_n<KC>(st.trow + colS, r);
                tc_wait_ld();
#pragma unroll
                for (int c = 0; c < NV; ++c) v[c] = __uint_as_float(r[c]);
                if (j * kKT + kKT > st.lim_all) {   // the causal edge or the chunk's end lies in this tile
#pragma unroll
                    for (int c = 0; c < NV; ++c)
                        if (k0 + c >= st.lim) v[c] = -INFINITY;
                }
            };
            uint32_t own[NV / 2];
            float psum;
            {
                float v[NV];
                load_scores(v);
                psum = exp_tile<NV>(v, st.mref, own);
            }
            // Every p of the tile is at most the tile's sum, so a sum within
            // kSumMax keeps each within fp16's range and the reference stands
            // without the tile's max. A row that sees a key of the chunk but
            // has no reference yet, or a larger sum (or a NaN), takes the warp
            // through the max: the scores are loaded again (S is still in
            // tensor memory), a row whose max rose takes it as the new
            // reference (O rescaled), and p is recomputed. (A lane without a
            // query, or a row that sees no key of the chunk, keeps -inf: its p
            // are 0.)
            const bool slow = (st.mref == -INFINITY && st.lim > 0) || !(psum <= kSumMax);
            if (__any_sync(0xFFFFFFFFu, slow)) {
                float v[NV];
                load_scores(v);
                float m4[4];   // four independent chains of three-input maxima
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    m4[a] = v[a];
#pragma unroll
                    for (int c = a + 4; c < NV; c += 8) m4[a] = max3f(m4[a], v[c], c + 4 < NV ? v[c + 4] : v[c]);
                }
                float mx = max3f(m4[0], m4[1], fmaxf(m4[2], m4[3]));
                if (DUAL) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));   // the row's two halves
                const float mxs = mx * kLog2e8;
                const bool resc = mxs > st.mref;
                if (__any_sync(0xFFFFFFFFu, resc)) {
                    // O holds P.V of the unit's tiles < j; the last of them (j-1) must be done
                    if (j >= 1 && !mbar_wait_warp(su32(&bars->o_done[(gj - 1) % kSBuf]), ((gj - 1) / kSBuf) & 1, st.abortp))
                        break;
                    tc_fence_after();
                    const float alpha = resc ? ex2(st.mref - mxs) : 1.f;
                    if (resc) {
                        st.mref = mxs;
                        st.l *= alpha;
                    }
                    if (j >= 1) {
                        if constexpr (DUAL) {   // this thread's 32 columns of O
#pragma unroll 1
                            for (int h = 0; h < 2; ++h) {
                                uint32_t o16[16];
                                tc_ld16x2_16<32>(st.trow + kColO + 16 * h, o16);
                                tc_wait_ld();
#pragma unroll
                                for (int c = 0; c < 16; ++c) o16[c] = __float_as_uint(__uint_as_float(o16[c]) * alpha);
                                tc_st16x2_16<32>(st.trow + kColO + 16 * h, o16);
                            }
                        } else {
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
                        }
                        tc_wait_st();
                    }
                }
                psum = exp_tile<NV>(v, st.mref, own);   // rows that kept their reference get the same values
            }
            if constexpr (DUAL) {   // P (fp16 pairs) of lane L: keys 0-31 at columns 0-15, 32-63 at 16-31
                tc_st16x2_16<KC / 4>(st.trow + colS, own);
            } else {
                tc_st_n<KC / 2>(st.trow + colS, own);
            }
            st.l += psum;
            tc_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(su32(&bars->p_full[b]));
    }
}

// The m-th unit the producer handed this CTA after its first (blockIdx.x), or
// -1: no more (or the CTA gave up). Single-thread consumer (the MMA thread).
__device__ __forceinline__ int next_unit_thread(Bars* bars, int m, volatile WaitCtl* abortp) {
    const int slot = m % kUQ;
    if (!mbar_wait(su32(&bars->uq_full[slot]), (m / kUQ) & 1, abortp)) return -1;
    const int u = reinterpret_cast<volatile int32_t*>(bars->uq)[slot];
    mbar_arrive(su32(&bars->uq_empty[slot]));
    return u;
}
// The same for a whole warp: every lane reads, then lane 0 releases the slot.
__device__ __forceinline__ int next_unit_warp(Bars* bars, int m, volatile WaitCtl* abortp) {
    const int slot = m % kUQ;
    int u = -1;
    if (mbar_wait_warp(su32(&bars->uq_full[slot]), (m / kUQ) & 1, abortp))
        u = reinterpret_cast<volatile int32_t*>(bars->uq)[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(su32(&bars->uq_empty[slot]));
    return u;
}

// The four softmax warps (128 threads) meet; bounded like every wait here.
__device__ __forceinline__ bool group_sync(Bars* bars, int& ph, volatile WaitCtl* abortp) {
    mbar_arrive(su32(&bars->grp));
    const bool ok = mbar_wait(su32(&bars->grp), ph & 1, abortp);
    ++ph;
    return ok;
}

// Query rows of a unit per TMEM lane quadrant: 16 for windows of at most 16
// rows (dual softmax: lanes L and L + 16 of a quadrant hold the same query),
// 32 for the prompt's wider windows. Quadrant w holds the unit's queries
// [per*w, per*w + per), i.e. window rows per/4*w .. +per/4 - 1 with their four
// heads of the KV head.
__device__ __forceinline__ int q_per(int rows) { return rows <= 16 ? 16 : 32; }

// The unit's queries into shared memory by TMA (one thread), K-major with the
// 128-byte swizzle, lane L of the Q tile holding query per*(L/32) + L%per
// (dual: lanes L%32 < 16 only): boxes of 16 query rows (4 window rows x 4
// heads), completing `bar` with 16 KB. Rows past the window belong to no query
// of the unit (other streams' rows, or zeros past the last row): their lanes
// are not valid rows and their results are never written.
__device__ __forceinline__ void issue_q(uint32_t sQ, const CUtensorMap* qmap, const Unit& U, uint32_t bar) {
    const bool dual = U.st.rows <= 16;
    mbar_expect_tx(bar, dual ? kQB / 2 : kQB);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int w = k >> 1, h = k & 1;
        // dual: lanes 0-15 of quadrant w hold window rows 4w..4w+3 (lanes 16-31
        // hold no query: their S rows are never read); else the halves hold
        // rows 8w..8w+3 and 8w+4..8w+7
        if (dual && h) continue;
        const int row = U.st.row_offset + (dual ? 4 * w : 8 * w + 4 * h);
        tma_load_3d(sQ + uint32_t(32 * w + 16 * h) * 128u, qmap, 0, 4 * U.g, row, bar);
    }
}

// The exact recompute of the units the launch queued (rare: V beyond fp16's
// range, or so small that fp16 would cost relative precision), by the last
// CTA's warps 0-3 (128 threads, named barrier 1) once every other CTA is done:
// each unit's window rows in groups of 8 (32 query rows) with the mma.sync
// item code on its exact path (V in bf16, P split into two bf16 parts),
// writing the unit's records or output again; then the unit's deferred merge
// arrival (a last-CTA merge runs here when it completes the count).
__device__ __noinline__ void recompute_exact(const SegTable& t, int layer, const uint16_t* q, float* part_o,
                                             float2* part_ml, float* out, int full, unsigned char* smem, int tid) {
    const int n = *reinterpret_cast<volatile const int32_t*>(t.tc_redo);
    __shared__ int last_flag;
    for (int k = 0; k < n; ++k) {
        const Unit U = unit_of(t, layer, __ldcg(t.tc_redo + 1 + k));
        const int mode = out ? U.st.merge_mode : kMergeKernel;
        for (int q0 = 0; q0 < 4 * U.st.rows; q0 += 32) {
            const AttnItem it{U.stream, U.chunk, q0, 0};
            item::attn_item<2, false, 1>(t, layer, it, U.st, U.g, q, part_o, part_ml, out, mode, full, smem, tid,
                                         false);
            item::bar_sync(1);   // the item's shared memory is reused by the next group
        }
        if (mode == kMergeLastCta) {
            __threadfence();
            item::bar_sync(1);
            int* ctr = t.counters + (size_t(layer) * t.S + U.stream) * TF_NKV + U.g;
            if (tid == 0) last_flag = atomicAdd(ctr, 1) == U.st.n_chunks - 1;
            item::bar_sync(1);
            if (last_flag) {
                __threadfence();
                merge_stream_head<4>(U.st, U.g, part_o, part_ml, out, tid, 128);
                if (tid == 0) atomicExch(ctr, 0);
            }
            item::bar_sync(1);
        }
    }
}

// Persistent: one launch of at most two CTAs per SM; each CTA runs its units
// back to back. A CTA starts with unit blockIdx.x; whenever its TMA producer
// has issued a unit's last tile it takes the next unit of the launch (an atomic
// counter in the table, so the largest-first list is handed out greedily) and
// passes it to the other roles through a small queue in shared memory. The
// TMA producer and the MMA thread run into the next unit's tiles while the
// softmax warps finish the previous unit (records, merges); the ring stages, S
// buffers and their mbarrier phases follow one running tile count.
__global__ void __launch_bounds__(kThreads, 2)
attn_partials_tc_kernel(SegTable t, int layer, const uint16_t* __restrict__ q, float* __restrict__ part_o,
                        float2* __restrict__ part_ml, float* __restrict__ out, int full, int n_units,
                        const __grid_constant__ CUtensorMap qmap) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = su32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;            // 128-byte swizzle atoms need 1 KB alignment
    unsigned char* gbase = smem_raw + (base - raw);
    const uint32_t sQ = base;
    const uint32_t sStage = base + kQB;
    Bars* bars = reinterpret_cast<Bars*>(gbase + kQB + kStages * kStageB);
    volatile WaitCtl* abortp = &bars->wc;
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
        mbar_init(su32(&bars->q_ready), 1);         // the q.K thread's expect_tx, then the TMA bytes
        mbar_init(su32(&bars->q_free), 1);          // the q.K thread's commit after a unit's last q.K
        for (int k = 0; k < kUQ; ++k) {
            mbar_init(su32(&bars->uq_full[k]), 1);
            mbar_init(su32(&bars->uq_empty[k]), kUQConsumers);
        }
        mbar_init(su32(&bars->grp), 128);
        mbar_init(su32(&bars->drain), 1);
        mbar_init(su32(&bars->drain_pv), 1);
        bars->wc.flag = 0;
        bars->wc.limit_ns = t.wait_ns;
        bars->redo_m = -1;
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        bars->alt = int32_t(atomicAdd(&g_tc_sm_launches[smid & 1023u], 1u) & 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid == 0 && int(blockIdx.x) < n_units) {   // the first unit's first tiles into L2 meanwhile
        const Unit U = unit_of(t, layer, blockIdx.x);
        for (int j = 0; j < U.T && j < kStages; ++j) {
            tma_prefetch_3d(U.kmap, 0, U.c0 + j * kKT, U.g);
            tma_prefetch_3d(U.vmap, 0, U.c0 + j * kKT, U.g);
        }
    }
    pdl_wait();   // the table above; queries and caches below
    if (warp == 4) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(su32(&bars->tmem_base)), "r"(kCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    // warp 5 converts V and warp 6 issues the TMA loads, or the other way round
    // (the two CTAs of an SM keep their converters on different sub-partitions)
    const int w_conv = bars->alt ? 6 : 5, w_prod = bars->alt ? 5 : 6;

    if (warp == 4) {
        // ------------------------------------------------------------ q.K MMAs
        // S(g) may be issued as soon as K tile g has landed and the P.V of tile
        // g-3 has released its S buffer, independently of the P.V thread, so
        // the scores stay ahead of the softmax
        if (lane == 0) {
            const uint64_t dq = sdesc(sQ, 16, 1024);
            bool ok = true;
            int gt = 0, n = 0, q_issued = 0;
            if (int(blockIdx.x) < n_units) {
                issue_q(sQ, &qmap, unit_of(t, layer, blockIdx.x), su32(&bars->q_ready));
                q_issued = 1;
            }
            for (int u = blockIdx.x; u >= 0 && ok; ++n) {
                const int T = unit_of(t, layer, u).T;
                ok = mbar_wait(su32(&bars->q_ready), n & 1, abortp);   // the unit's queries landed
                if (!ok) break;
                tc_fence_after();
                for (int j = 0; j < T && ok; ++j) {
                    const int g1 = gt + j, s = g1 % kStages, b = g1 % kSBuf;
                    ok = mbar_wait(su32(&bars->kv_full[s]), (g1 / kStages) & 1, abortp);
                    if (!ok) break;
                    if (g1 >= kSBuf) {   // P.V(g1-3) has released S buffer b
                        ok = mbar_wait(su32(&bars->o_done[b]), ((g1 - kSBuf) / kSBuf) & 1, abortp);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    const uint64_t dk = sdesc(sStage + s * kStageB, 16, 1024);
#pragma unroll
                    for (int k = 0; k < TF_D / 16; ++k)   // K = 64: 4 steps of 16 (32 bytes)
                        tc_mma_ss(tmem + kColS + 64 * b, dq + 2 * k, dk + 2 * k, kIdescQK, k > 0 ? 1u : 0u);
                    tc_commit(su32(&bars->s_full[b]));
                }
                gt += T;
                if (!ok) break;
                // the next unit's queries, as soon as this unit's q.K have read the
                // buffer (long before the softmax finishes this unit)
                tc_commit(su32(&bars->q_free));
                u = next_unit_thread(bars, n, abortp);
                if (u >= 0) {
                    ok = mbar_wait(su32(&bars->q_free), n & 1, abortp);
                    if (ok) {
                        issue_q(sQ, &qmap, unit_of(t, layer, u), su32(&bars->q_ready));
                        ++q_issued;
                    }
                }
            }
            tc_commit(su32(&bars->drain));   // every MMA this thread issued
            mbar_drain(su32(&bars->drain), 0);
            if (q_issued > n)   // a query load not waited for (the CTA gave up): let it land
                mbar_drain(su32(&bars->q_ready), (q_issued - 1) & 1);
        }
        __syncwarp();
    } else if (warp == 7) {
        // ------------------------------------------------------------ P.V MMAs
        if (lane == 0) {
            bool ok = true;
            int gt = 0, n = 0;
            for (int u = blockIdx.x; u >= 0 && ok; ++n) {
                const int T = unit_of(t, layer, u).T;
                for (int j = 0; j < T && ok; ++j) {
                    const int g2 = gt + j, s = g2 % kStages, b = g2 % kSBuf;
                    ok = mbar_wait(su32(&bars->p_full[b]), (g2 / kSBuf) & 1, abortp);
                    if (!ok) break;
                    ok = mbar_wait(su32(&bars->v_ready[s]), (g2 / kStages) & 1, abortp);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t dv = sdesc(sStage + s * kStageB + kTileB, kTileB, 1024);
#pragma unroll
                    for (int k = 0; k < kKT / 16; ++k)   // 64 keys: 4 steps of 16 (2 KB of V rows)
                        tc_mma_ts(tmem + kColO, tmem + kColS + 64 * b + 8 * k, dv + 128 * k, kIdescPV,
                                  (j > 0 || k > 0) ? 1u : 0u);
                    // the stage's K was read by the q.K of this tile, which completed
                    // before the softmax read S; V by this P.V
                    tc_commit(su32(&bars->o_done[b]));
                    tc_commit(su32(&bars->kv_empty[s]));
                }
                gt += T;
                if (ok) u = next_unit_thread(bars, n, abortp);
            }
            tc_commit(su32(&bars->drain_pv));
            mbar_drain(su32(&bars->drain_pv), 0);
        }
        __syncwarp();
    } else if (warp == w_prod) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            // K/V are read once: ask L2 to evict them first (measured 4% faster
            // than the default policy on the 64 x 16-row round)
            const uint64_t once = l2_evict_first();
            int gt = 0;
            bool ok = true;
            for (int u = blockIdx.x, m = 0; u >= 0 && ok; ++m) {
                const Unit U = unit_of(t, layer, u);
                for (int j = 0; j < U.T; ++j, ++gt) {
                    const int s = gt % kStages;
                    if (gt >= kStages &&   // the stage is free once the P.V of tile gt - kStages completed
                        !mbar_wait(su32(&bars->kv_empty[s]), ((gt - kStages) / kStages) & 1, abortp)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bar = su32(&bars->kv_full[s]);
                    mbar_expect_tx(bar, kStageB);
                    tma_load_3d_hint(sStage + s * kStageB, U.kmap, 0, U.c0 + j * kKT, U.g, bar, once);
                    tma_load_3d_hint(sStage + s * kStageB + kTileB, U.vmap, 0, U.c0 + j * kKT, U.g, bar, once);
                }
                if (!ok) break;
                // the next unit of the launch, for this CTA's roles
                int un = int(gridDim.x) + atomicAdd(&t.tc_work[2 * layer], 1);
                if (un >= n_units) un = -1;
                const int slot = m % kUQ;
                if (m >= kUQ && !mbar_wait(su32(&bars->uq_empty[slot]), ((m / kUQ) - 1) & 1, abortp)) break;
                bars->uq[slot] = un;
                mbar_arrive(su32(&bars->uq_full[slot]));   // release: the index is visible to the waiters
                u = un;
            }
            if (abortp->flag)   // let the copies in flight land before the CTA exits
                for (int k = gt > kStages ? gt - kStages : 0; k < gt; ++k)
                    mbar_drain(su32(&bars->kv_full[k % kStages]), (k / kStages) & 1);
        }
        __syncwarp();
    } else if (warp == w_conv) {
        // ------------------------------------------------------------ V tiles bf16 -> fp16
        int gt = 0;
        bool ok = true;
        for (int u = blockIdx.x, m = 0; u >= 0 && ok; ++m) {
            const int T = unit_of(t, layer, u).T;
            for (int j = 0; j < T; ++j, ++gt) {
                const int s = gt % kStages;
                if (!mbar_wait_warp(su32(&bars->kv_full[s]), (gt / kStages) & 1, abortp)) {
                    ok = false;
                    break;
                }
                const uint32_t vs = sStage + s * kStageB + kTileB + uint32_t(lane) * 16u;
                // all 16 loads first: one shared-memory round trip a tile, not
                // one per 16 bytes (the volatile loads and stores keep their order)
                constexpr int NC = kTileB / 16 / 32;
                uint4 v[NC];
#pragma unroll
                for (int c = 0; c < NC; ++c) v[c] = lds128(vs + uint32_t(32 * c) * 16u);
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    v[c].x = bf2_to_h2(v[c].x);
                    v[c].y = bf2_to_h2(v[c].y);
                    v[c].z = bf2_to_h2(v[c].z);
                    v[c].w = bf2_to_h2(v[c].w);
                    sts128(vs + uint32_t(32 * c) * 16u, v[c]);
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(su32(&bars->v_ready[s]));
                // the stage is refilled only after this tile's P.V, which waits on
                // this arrival, so the next use of this stage cannot overtake it
            }
            if (ok) u = next_unit_warp(bars, m, abortp);
        }
    } else {
        // ------------------------------------------------------------ softmax + records
        int gt = 0, gph = 0;
        const uint32_t trow = tmem + (uint32_t(warp * 32) << 16);
        for (int u = blockIdx.x, m = 0; u >= 0; ++m) {
            const Unit U = unit_of(t, layer, u);
            const SegStream& st = U.st;
            const int nq = st.rows * 4, per = q_per(st.rows);
            const bool dual = per == 16;
            const int ql = dual ? (lane & 15) : lane;   // the lane's query within the quadrant
            const int qi = per * warp + ql;
            const bool qvalid = ql < per && qi < nq;
            const bool wact = per * warp < nq;      // the warp holds at least one real row
            const int mode = out ? st.merge_mode : kMergeKernel;   // records only in the two-call form
            SoftState ss;
            ss.bars = bars;
            ss.abortp = abortp;
            ss.trow = trow;
            ss.g0 = gt;
            ss.T = U.T;
            // chunk-local key bounds: causal count of the row (of row 0 for lim_all),
            // or every key for a FULL block
            ss.lim = qvalid ? (full ? st.keys : st.keys - st.rows + (qi >> 2) + 1) - U.c0 : 0;
            ss.lim_all = (full ? st.keys : st.keys - st.rows + 1) - U.c0;
            ss.wact = wact;
            ss.mref = -INFINITY;
            ss.l = 0.f;
            if (dual)
                softmax_tiles<kKT, true>(ss);
            else
                softmax_tiles<kKT, false>(ss);
            gt += U.T;
            const int un = next_unit_warp(bars, m, abortp);
            if (!abortp->flag) mbar_wait(su32(&bars->o_done[(gt - 1) % kSBuf]), ((gt - 1) / kSBuf) & 1, abortp);
            tc_fence_after();
            if (wact) {
                // (m, l, O) relative to the row's reference max -> the chunk's record
                // (the merge weighs each record by 2^(m - M): any reference the
                // p were taken against gives the same result)
                const bool aborted = abortp->flag != 0;
                const float f = 1.f;
                // this thread's columns of O: all 64 of its lane, or (dual) its
                // half [d0, d0 + 32) of lane L's row
                auto finish = [&](auto& ro) {
                    constexpr int ND = int(sizeof(ro) / sizeof(ro[0]));
                    const int d0 = ND == 32 ? 32 * (lane >> 4) : 0;
                    float lsum = ss.l;
                    if (ND == 32) lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 16);   // the row's two key halves
                    // P.V ran with V in fp16. A row whose O is not finite (a V of
                    // 65,536 or more has no fp16 value), or a warp whose rows'
                    // outputs |o| / l all lie below 2^-10 (fp16's subnormal steps
                    // of 2^-24 would cost relative precision), sends the unit to
                    // the exact recompute at the end of the launch; its records
                    // are rewritten there and its merge waits for them.
                    bool nonfinite = false, big = false;
                    if (qvalid && lsum > 0.f) {
                        nonfinite = !isfinite(lsum);
#pragma unroll
                        for (int c = 0; c < ND; ++c) {
                            const float v = __uint_as_float(ro[c]);
                            nonfinite |= !isfinite(v);
                            big |= fabsf(v) >= 0x1p-10f * lsum;
                        }
                    }
                    const bool seen = __any_sync(0xFFFFFFFFu, qvalid && lsum > 0.f);
                    const bool redo = !aborted && (__any_sync(0xFFFFFFFFu, nonfinite) ||
                                                   (seen && !__any_sync(0xFFFFFFFFu, big)));
                    if (redo && lane == 0 && atomicMax(&bars->redo_m, m) < m)
                        t.tc_redo[1 + atomicAdd(t.tc_redo, 1)] = u;
                    if (qvalid && mode == kMergeDirect) {   // the stream's only chunk: the output itself
                        const float inv = aborted ? NAN : 1.f / lsum;   // a row always sees key 0 of its stream
                        float4* dst = reinterpret_cast<float4*>(out_row(out, st, U.g, qi) + d0);
#pragma unroll
                        for (int c = 0; c < ND / 4; ++c)
                            dst[c] = make_float4(__uint_as_float(ro[4 * c]) * inv,
                                                 __uint_as_float(ro[4 * c + 1]) * inv,
                                                 __uint_as_float(ro[4 * c + 2]) * inv,
                                                 __uint_as_float(ro[4 * c + 3]) * inv);
                    } else if (qvalid) {
                        const int64_t rec = st.pbase + (int64_t(U.chunk) * TF_NKV + U.g) * nq + qi;
                        const bool empty = ss.mref == -INFINITY;
                        float4* dst = reinterpret_cast<float4*>(part_o + rec * TF_D + d0);
#pragma unroll
                        for (int c = 0; c < ND / 4; ++c) {
                            float4 v = make_float4(__uint_as_float(ro[4 * c]) * f, __uint_as_float(ro[4 * c + 1]) * f,
                                                   __uint_as_float(ro[4 * c + 2]) * f,
                                                   __uint_as_float(ro[4 * c + 3]) * f);
                            if (aborted) v = make_float4(NAN, NAN, NAN, NAN);
                            else if (empty) v = make_float4(0.f, 0.f, 0.f, 0.f);
                            dst[c] = v;
                        }
                        if (d0 == 0)
                            part_ml[rec] = aborted ? make_float2(NAN, INFINITY)
                                                   : make_float2(ss.mref, empty ? 0.f : lsum * f);
                    }
                };
                if (dual) {
                    uint32_t r32[32];
                    tc_ld16x2_32<32>(trow + kColO, r32);
                    tc_wait_ld();
                    finish(r32);
                } else {
                    uint32_t r64[64];
                    tc_ld64(trow + kColO, r64);
                    tc_wait_ld();
                    finish(r64);
                }
            }
            // O is read: the next unit's first P.V (which overwrites it) waits for
            // this thread's next p_full arrival
            tc_fence_before();
            if (mode == kMergeLastCta) {
                // every CTA of (stream, KV head) counts its arrival after its records
                // are visible; the last one merges and resets the counter
                __threadfence();
                if (group_sync(bars, gph, abortp)) {
                    int* ctr = t.counters + (size_t(layer) * t.S + U.stream) * TF_NKV + U.g;
                    // a unit queued for the exact recompute arrives after it
                    if (tid == 0)
                        bars->last = *reinterpret_cast<volatile int32_t*>(&bars->redo_m) == m
                                         ? 0 : (atomicAdd(ctr, 1) == st.n_chunks - 1);
                    if (group_sync(bars, gph, abortp) && bars->last) {
                        __threadfence();
                        merge_stream_head<2, 4>(st, U.g, part_o, part_ml, out, tid, 128);
                        if (tid == 0) atomicExch(ctr, 0);
                    }
                }
            }
            u = un;
        }
    }
    tc_fence_before();
    __syncthreads();   // every role is done
    tc_fence_after();
    if (tid == 0) {
        // a CTA that gave up a wait reports it in the table's status word
        // (tf_segments_status reads it and resets the table's counters)
        if (abortp->flag) atomicOr(t.status, uint32_t(TF_STATUS_ATTN_TIMEOUT));
        // the last CTA to finish (every unit has been handed out by then) resets
        // the work counters for the next launch and runs the exact recomputes
        __threadfence();
        const bool last = atomicAdd(&t.tc_work[2 * layer + 1], 1) == int(gridDim.x) - 1;
        if (last) {
            atomicExch(&t.tc_work[2 * layer], 0);
            atomicExch(&t.tc_work[2 * layer + 1], 0);
        }
        bars->is_last = last ? 1 : 0;
    }
    pdl_trigger();
    if (warp == 4) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
    }
    __syncthreads();
    if (bars->is_last) {
        __threadfence();   // every CTA queued its units before it counted itself done
        if (warp < 4) recompute_exact(t, layer, q, part_o, part_ml, out, full, gbase, tid);
        __syncthreads();
        if (tid == 0) t.tc_redo[0] = 0;
    }
}

}  // namespace

int attn_tc_prepare() {
    cudaError_t e = cudaFuncSetAttribute(attn_partials_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    return e == cudaSuccess ? TF_OK : cuda_fail(e);
}

int launch_attn_partials_tc(const SegTable& t0, int layer, const uint16_t* q, float* po, float2* pml,
                            cudaStream_t stream, float* out, int full, int grid_cap) {
    if (!t0.k_maps || !t0.v_maps) return TF_EINVAL;
    SegTable t = t0;
    t.wait_ns = wait_limit_ns();
    const int n_units = (t.n_items - t.n_items_mma) * TF_NKV;
    const int slots = grid_cap > 0 ? grid_cap : 2 * sm_count();   // two CTAs per SM, all resident
    const int grid = n_units < slots ? n_units : slots;
    CUtensorMap qmap;
    if (!encode_q_map(&qmap, q, t.R)) return cuda_fail(cudaErrorInvalidValue);
    return launch_pdl(attn_partials_tc_kernel, dim3(grid), dim3(kThreads), kSmemBytes, stream, t, layer, q, po, pml,
                      out, full, n_units, qmap);
}

}  // namespace tf
