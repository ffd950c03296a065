// The drafter's Markov head on the 5th-generation tensor cores: per block row,
// score[v] = bf16(base[v] + bf16(W2[v] . W1[tok])) over the vocabulary and the
// lowest token of the largest score, step after step (one block row of every
// stream a step): the whole chain in one cooperative launch for tables of up
// to 128 streams (markov_chain_kernel, at the end of this file), else one
// launch a step (markov_step_kernel, described here).
//
// PR #1391 "lfm2: draft with LiquidAI's DSpark drafter (--drafter)": the head
// adds to each draft row's logits the product of W2 with the W1 row of the
// previous pick and takes the argmax, row by row in sequence; its kernels do
// the W1 gather, the W2 dot, the add and an argmax that takes the lowest token
// on a tie and flags a NaN score; the family test states the step as the
// argmax of bf16(base + bf16(W2 . W1[prev])); W2 is scanned in bf16.
//
// One step is a skinny GEMM followed by an argmax: D[s][v] = E[s] . W2[v] with
// E[s] = W1[tok_s], for up to 128 streams (MMA M = 128 TMEM lanes, one lane per
// stream; lanes without a stream hold zero rows; stream L of the group sits on
// lane 32*(L%4) + L/4, so a few streams still spread over all four lane
// quadrants and their epilogue warps) against 128-row tiles of W2
// (MMA N = 128), K = 256. W2 is 128000 x 512 bytes and is read once per step
// for all the streams, so the step is HBM bound on W2 plus each stream's base
// row; the tensor cores keep the 2*128*256 flops per W2 row off the ALUs.
//
// CTA (one per SM; a contiguous range of W2 tiles), 6 warps:
//   warp 5, lane 0   TMA loads of W2 k-blocks (128 rows x 64 columns = 16 KB,
//                    128-byte swizzle) into an 8-stage ring;
//   warp 4, lane 0   the MMAs: 4 per k-block, into one of two 128-column
//                    accumulators in tensor memory (tile t uses t % 2);
//   warps 0-3        epilogue: thread = stream lane; per tile it reads its 128
//                    dot products, rounds them to bf16 two at a time
//                    (cvt.rn.bf16x2.f32), adds its stream's base logits
//                    (add.rn.bf16x2: one rounding of the exact sum; the base is
//                    loaded a tile ahead), tests the exponents for nonfinite
//                    scores and takes the packed maximum of each 32 columns;
//                    only when that maximum beats the running best does it
//                    look for the first column holding it -- the argmax is
//                    within the thread, no shuffles.
// The CTAs of a launch meet through 64-bit atomicMax on (ordered score, ~token)
// per stream and an atomicOr of the flags; the last CTA to finish writes the
// picks and resets the scratch. The next step's launch reads those picks as
// its previous tokens.
//
// Every mbarrier wait is bounded (the library's wait limit, 2 s of
// %globaltimer unless tf_set_wait_limit_ns changed it); on a timeout the CTA
// raises its abort flag, drains its copies and MMAs (bounded), marks its
// streams' rows with flag bit 1, sets TF_STATUS_MARKOV_TIMEOUT in the table's
// status word, frees its tensor memory and returns.
#include <cstdlib>
#include <cstring>

#include "tc_ptx.cuh"

namespace tf {
namespace {

constexpr int kLanes = 128;             // streams per group: MMA M, TMEM lanes
constexpr int kTileV = 128;             // W2 rows per tile: MMA N
constexpr int kKB = TF_MK / 64;         // k-blocks of 64 columns (128 bytes) per row
constexpr int kSlabB = 128 * 128;       // one k-block of 128 rows: 16 KB
constexpr int kStages = 8;
constexpr int kAB = kKB * kSlabB;       // E: 128 rows x 256 columns, 64 KB
constexpr int kWarps = 6;
constexpr int kThreads = kWarps * 32;
constexpr uint32_t kCols = 256;         // two accumulators of 128 columns

// TMEM lane (= row of E) of the group's stream L, and back
__host__ __device__ constexpr int lane_of(int L) { return 32 * (L & 3) + (L >> 2); }

struct Bars {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    WaitCtl wc;             // abort flag and wait limit of the CTA's bounded waits
    int32_t last;
    int32_t tok[kLanes];    // previous token of the lane's stream, -1 if none or invalid
    int32_t row[kLanes];    // draft row of the lane's stream in this step, -1 if it has none
};
constexpr int kSmemBytes = 1024 + kAB + kStages * kSlabB + int(sizeof(Bars));

// kind::f16, fp32 accumulate, A and B bf16 K-major, N = 128, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(kTileV >> 3) << 17) |
                            (uint32_t(128 >> 4) << 24);

// Orders scores as unsigned integers (larger score -> larger key); -0 is +0.
__device__ __forceinline__ uint32_t ord_bf16(float best) {
    uint32_t b = best == 0.f ? 0u : (__float_as_uint(best) >> 16);
    return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}

// The base logits of columns [v0, v0 + 2*NW) of a row as NW bf16 pairs, zeros
// past the vocabulary (v0 a multiple of 8). The branch depends on the tile
// alone (uniform across the threads that share it).
template <int NW>
__device__ __forceinline__ void load_base(const uint16_t* brow, int v0, int vocab, uint32_t (&dst)[NW]) {
    if (v0 + 2 * NW <= vocab) {
        const uint4* bp = reinterpret_cast<const uint4*>(brow + v0);
#pragma unroll
        for (int k = 0; k < NW / 4; ++k) {
            const uint4 x = __ldcs(bp + k);   // read once: evict first
            dst[4 * k] = x.x;
            dst[4 * k + 1] = x.y;
            dst[4 * k + 2] = x.z;
            dst[4 * k + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const int i0 = v0 + 2 * k;
            const uint32_t lo = i0 < vocab ? brow[i0] : 0u;
            const uint32_t hi = i0 + 1 < vocab ? brow[i0 + 1] : 0u;
            dst[k] = lo | (hi << 16);
        }
    }
}
// The 128 base logits of one tile of the lane's row.
__device__ __forceinline__ void load_base_tile(const uint16_t* brow, int v0, int vocab, uint32_t (&dst)[64]) {
    load_base<64>(brow, v0, vocab, dst);
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// {hi, lo} fp32 -> bf16 pair, each rounded to nearest even
__device__ __forceinline__ uint32_t cvt_bf16x2(float hi, float lo) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
// bf16 pair sum, each the exact sum rounded once to nearest even
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 32 scores as 16 bf16 pairs, by value, for the out-of-line paths below.
struct Pairs16 {
    uint32_t w[16];
};
// Columns [n, 32) lie past the vocabulary: the most negative finite value
// there (never first, never flagged). Out of line: only the vocabulary's last
// tile takes it, and the hot loops stay small enough for the instruction cache.
__device__ __noinline__ Pairs16 mask_past_vocab(Pairs16 sc, int n) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        if (2 * k >= n) sc.w[k] = (sc.w[k] & 0xFFFF0000u) | 0xFF7Fu;
        if (2 * k + 1 >= n) sc.w[k] = (sc.w[k] & 0x0000FFFFu) | 0xFF7F0000u;
    }
    return sc;
}
// The first of the 32 columns holding mv (out of line: taken only when the
// running best improves, a few times a step).
__device__ __noinline__ int first_column(Pairs16 sc, float mv) {
    int c = 31;
#pragma unroll
    for (int k = 15; k >= 0; --k) {
        if (bf_hi(sc.w[k]) == mv) c = 2 * k + 1;
        if (bf_lo(sc.w[k]) == mv) c = 2 * k;
    }
    return c;
}

// The scores of 32 columns as 16 bf16 pairs (ids v .. v+31, `n` of them
// inside the vocabulary): nonfinite bits and the running first largest.
__device__ __forceinline__ void score_sums(uint32_t (&sc)[16], int v, int n, float& best, int& bid, uint32_t& nf) {
    if (n < 32) {
        Pairs16 p;
#pragma unroll
        for (int k = 0; k < 16; ++k) p.w[k] = sc[k];
        p = mask_past_vocab(p, n);
#pragma unroll
        for (int k = 0; k < 16; ++k) sc[k] = p.w[k];
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) nf |= (sc[k] & 0x7F807F80u) + 0x00800080u;   // bit 15 / 31: exponent all ones
    uint32_t m8[8], m4[4];
#pragma unroll
    for (int k = 0; k < 8; ++k) m8[k] = max_bf16x2(sc[2 * k], sc[2 * k + 1]);
#pragma unroll
    for (int k = 0; k < 4; ++k) m4[k] = max_bf16x2(m8[2 * k], m8[2 * k + 1]);
    const uint32_t m = max_bf16x2(max_bf16x2(m4[0], m4[1]), max_bf16x2(m4[2], m4[3]));
    const float mv = fmaxf(bf_lo(m), bf_hi(m));
    if (mv > best) {   // rare after the first tiles: find the first column holding mv
        Pairs16 p;
#pragma unroll
        for (int k = 0; k < 16; ++k) p.w[k] = sc[k];
        bid = v + first_column(p, mv);
        best = mv;
    }
}
// 32 columns from their fp32 dot products: each rounded to bf16, plus the base.
__device__ __forceinline__ void score_piece(const uint32_t (&r)[32], const uint32_t* base16, int v, int n,
                                            float& best, int& bid, uint32_t& nf) {
    uint32_t sc[16];
#pragma unroll
    for (int k = 0; k < 16; ++k)
        sc[k] = add_bf16x2(cvt_bf16x2(__uint_as_float(r[2 * k + 1]), __uint_as_float(r[2 * k])), base16[k]);
    score_sums(sc, v, n, best, bid, nf);
}

__global__ void __launch_bounds__(kThreads, 1)
markov_step_kernel(SegTable t, int step, const uint16_t* __restrict__ W1, int vocab,
                   const uint16_t* __restrict__ base, int64_t base_stride, const int32_t* __restrict__ prev,
                   int32_t* __restrict__ pick, uint8_t* __restrict__ flag,
                   const __grid_constant__ CUtensorMap w2map) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = su32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;          // 128-byte swizzle atoms need 1 KB alignment
    unsigned char* gbase = smem_raw + (sbase - raw);
    const uint32_t sA = sbase;
    const uint32_t sB = sbase + kAB;
    Bars* bars = reinterpret_cast<Bars*>(gbase + kAB + kStages * kSlabB);
    volatile WaitCtl* abortp = &bars->wc;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int group = blockIdx.y;
    const int s0 = group * kLanes;
    const int nt = (vocab + kTileV - 1) / kTileV;
    const int t_begin = int((int64_t(blockIdx.x) * nt) / gridDim.x);
    const int t_end = int((int64_t(blockIdx.x + 1) * nt) / gridDim.x);
    const int ntl = t_end - t_begin;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(su32(&bars->full[s]), 1);
            mbar_init(su32(&bars->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(su32(&bars->acc_full[b]), 1);
            mbar_init(su32(&bars->acc_empty[b]), 4);   // the 4 epilogue warps
        }
        mbar_init(su32(&bars->drain), 1);
        bars->wc.flag = 0;
        bars->wc.limit_ns = t.wait_ns;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_wait();   // previous tokens may be the picks of the step just before
    if (tid < kLanes) {
        const int s = s0 + tid;
        int tok = -1, row = -1;
        if (s < t.S) {
            const SegStream st = t.streams[s];
            if (st.rows - 1 > step) {
                row = st.row_offset - s + step;
                tok = step == 0 ? prev[s] : pick[row - 1];
                if (tok < 0 || tok >= vocab) tok = -1;
            }
        }
        bars->tok[tid] = tok;
        bars->row[tid] = row;
    }
    if (warp == 4) tc_alloc(su32(&bars->tmem_base), kCols);
    __syncthreads();
    // E = the streams' W1 rows (zero rows for lanes without a token), K-major,
    // 128-byte swizzled: 16-byte chunk c of row m in k-block c / 8. Every copy
    // is in flight at once (cp.async), then one wait.
    for (int idx = tid; idx < kLanes * (TF_MK / 8); idx += kThreads) {
        const int L = idx >> 5, c = idx & 31, m = lane_of(L);
        const int tok = bars->tok[L];
        const uint16_t* src = tok >= 0 ? W1 + size_t(tok) * TF_MK + c * 8 : W1;
        cp_async16(sA + (c >> 3) * kSlabB + m * 128 + (((c & 7) ^ (m & 7)) << 4), src, tok >= 0);
    }
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    float best = -INFINITY;
    int bid = 0x7FFFFFFF;
    uint32_t nf = 0;
    const int L = 4 * lane + warp;   // the stream on TMEM lane 32*warp + lane (epilogue warps)
    const int my_tok = warp < 4 ? bars->tok[L] : -1;
    const int my_row = warp < 4 ? bars->row[L] : -1;

    if (warp == 5) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            // W2 is read again by every step of the chain: ask L2 to keep it
            // (the base rows, read once, stream past it)
            const uint64_t keep = l2_evict_last();
            int issued = 0;
            for (int i = 0; i < ntl * kKB; ++i) {
                const int s = i % kStages;
                if (i >= kStages && !mbar_wait(su32(&bars->empty[s]), ((i / kStages) - 1) & 1, abortp)) break;
                const uint32_t bar = su32(&bars->full[s]);
                mbar_expect_tx(bar, kSlabB);
                tma_load_2d_hint(sB + s * kSlabB, &w2map, (i % kKB) * 64, (t_begin + i / kKB) * kTileV, bar, keep);
                ++issued;
            }
            if (abortp->flag)   // let the copies in flight land before the CTA exits
                for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
                    mbar_drain(su32(&bars->full[i % kStages]), (i / kStages) & 1);
        }
        __syncwarp();
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            bool ok = true;
            for (int tt = 0; tt < ntl && ok; ++tt) {
                const int b = tt & 1;
                if (tt >= 2) {   // the epilogue has read this accumulator's previous tile
                    ok = mbar_wait(su32(&bars->acc_empty[b]), ((tt >> 1) - 1) & 1, abortp);
                    if (!ok) break;
                }
                tc_fence_after();
                for (int kb = 0; kb < kKB && ok; ++kb) {
                    const int i = tt * kKB + kb, s = i % kStages;
                    ok = mbar_wait(su32(&bars->full[s]), (i / kStages) & 1, abortp);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t da = sdesc(sA + kb * kSlabB, 16, 1024);
                    const uint64_t db = sdesc(sB + s * kSlabB, 16, 1024);
#pragma unroll
                    for (int k = 0; k < 4; ++k)   // 64 columns: 4 steps of 16 (32 bytes)
                        tc_mma_ss(tmem + uint32_t(b * kTileV), da + 2 * k, db + 2 * k, kIdesc, (kb | k) ? 1u : 0u);
                    tc_commit(su32(&bars->empty[s]));   // the stage is free once these MMAs complete
                }
                if (ok) tc_commit(su32(&bars->acc_full[b]));
            }
            tc_commit(su32(&bars->drain));   // every MMA issued so far
            mbar_drain(su32(&bars->drain), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const bool valid = my_tok >= 0;
        const bool wact = __any_sync(0xFFFFFFFFu, valid);
        // lanes without a row read row 0 (any row exists when the kernel runs) and discard it
        const uint16_t* brow = base + (valid ? my_row : 0) * base_stride;
        const uint32_t tlane = tmem + (uint32_t(warp * 32) << 16);
        // base logits one tile ahead of the accumulator they are added to
        uint32_t cur[64], nxt[64];
        if (wact && ntl > 0) load_base_tile(brow, t_begin * kTileV, vocab, cur);
        for (int tt = 0; tt < ntl; ++tt) {
            const int b = tt & 1;
            const int v0 = (t_begin + tt) * kTileV;
            if (wact && tt + 1 < ntl) load_base_tile(brow, v0 + kTileV, vocab, nxt);
            if (!mbar_wait_warp(su32(&bars->acc_full[b]), (tt >> 1) & 1, abortp)) break;
            tc_fence_after();
            if (wact) {
#pragma unroll
                for (int p = 0; p < kTileV / 32; ++p) {
                    const int v = v0 + 32 * p;
                    if (v < vocab) {   // uniform
                        uint32_t r[32];
                        tc_ld_n<32>(tlane + uint32_t(b * kTileV + 32 * p), r);
                        tc_wait_ld();
                        const int n = vocab - v < 32 ? vocab - v : 32;
                        if (valid) score_piece(r, cur + 16 * p, v, n, best, bid, nf);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(su32(&bars->acc_empty[b]));
#pragma unroll
            for (int k = 0; k < 64; ++k) cur[k] = nxt[k];
        }
        nf = (nf & 0x80008000u) ? 1u : 0u;
    }
    tc_fence_before();
    __syncthreads();   // every copy and MMA of the CTA is done
    tc_fence_after();
    pdl_trigger();

    // this CTA's best of each stream, met across CTAs in the table's scratch
    if (warp < 4 && my_tok >= 0) {
        const int s = s0 + L;
        if (abortp->flag) {
            atomicOr(&t.mk_flags[s], 2u);
        } else {
            if (bid != 0x7FFFFFFF)
                atomicMax(&t.mk_keys[s], (static_cast<unsigned long long>(ord_bf16(best)) << 32) |
                                             static_cast<unsigned long long>(0xFFFFFFFFu - uint32_t(bid)));
            if (nf) atomicOr(&t.mk_flags[s], 1u);
        }
        __threadfence();
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        bars->last = atomicAdd(&t.mk_ctr[group], 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (bars->last) {
        // the last CTA of the group: picks and flags, then the scratch back to zero
        __threadfence();
        if (tid < kLanes && bars->row[tid] >= 0) {
            const int s = s0 + tid;
            const unsigned long long key = atomicExch(&t.mk_keys[s], 0ull);
            const uint32_t fl = atomicExch(&t.mk_flags[s], 0u);
            int p = -1;
            uint8_t f = 1;
            if (bars->tok[tid] >= 0) {
                if (fl) {
                    f = uint8_t(fl);
                } else {
                    p = int(0xFFFFFFFFu - uint32_t(key & 0xFFFFFFFFull));
                    f = 0;
                }
            }
            pick[bars->row[tid]] = p;
            flag[bars->row[tid]] = f;
        }
        if (tid == 0) atomicExch(&t.mk_ctr[group], 0u);
    }
    __syncthreads();
    if (tid == 0 && abortp->flag) atomicOr(t.status, uint32_t(TF_STATUS_MARKOV_TIMEOUT));
    if (warp == 4) {
        tc_fence_after();
        tc_dealloc(tmem, kCols);
    }
}

// ---- the whole chain in one launch --------------------------------------
//
// Tables of at most 128 streams (one lane group) run every step of the chain
// in one cooperative launch: the CTAs (one per SM, all resident) keep their
// range of W2 tiles for every step, the TMA producer streams those tiles step
// after step without a break (W2 does not depend on the picks), and between
// steps the CTAs meet once: each adds its best scores to the step's per-stream
// keys, counts its arrival, and the last to arrive writes the step's picks and
// opens the next step (a generation word); the epilogue warps then gather the
// next step's W1 rows while the producer is already filling the ring. Every
// wait is bounded: an mbarrier wait or the step barrier that runs out raises
// the CTA's abort flag and a global one (the other CTAs stop waiting), and the
// rows of the steps not done are flagged (bit 1).

struct ChainBars {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t e_ready;       // the step's W1 rows are in E (the 128 epilogue threads)
    uint64_t drain;
    uint32_t tmem_base;
    WaitCtl wc;             // abort flag and wait limit of the CTA's bounded waits
    int32_t last;
    int32_t stop;           // epilogue thread 0's snapshot of the abort flag, read after a barrier
    int32_t tok[kLanes];
    int32_t row[kLanes];
};
constexpr int kChainSmemBytes = 1024 + kAB + kStages * kSlabB + int(sizeof(ChainBars));

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Wait until the step barrier's generation reaches `target` (one thread).
__device__ bool chain_wait(const uint32_t* sync, uint32_t target, volatile WaitCtl* abortp) {
    const unsigned long long t0 = gtime(), limit = abortp->limit_ns;
    for (;;) {
        uint32_t g;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(g) : "l"(sync + 1) : "memory");
        if (g >= target) return true;
        if (abortp->flag) return false;
        if (*reinterpret_cast<const volatile uint32_t*>(sync + 2)) {   // another CTA gave up
            abortp->flag = 1;
            return false;
        }
        if (gtime() - t0 > limit) {
            abortp->flag = 1;
            return false;
        }
        __nanosleep(64);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
markov_chain_kernel(SegTable t, int steps, const uint16_t* __restrict__ W1, int vocab,
                    const uint16_t* __restrict__ base, int64_t base_stride, const int32_t* __restrict__ prev,
                    int32_t* __restrict__ pick, uint8_t* __restrict__ flag,
                    const __grid_constant__ CUtensorMap w2map) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = su32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    unsigned char* gbase = smem_raw + (sbase - raw);
    const uint32_t sA = sbase;
    const uint32_t sB = sbase + kAB;
    ChainBars* bars = reinterpret_cast<ChainBars*>(gbase + kAB + kStages * kSlabB);
    volatile WaitCtl* abortp = &bars->wc;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nt = (vocab + kTileV - 1) / kTileV;
    const int t_begin = int((int64_t(blockIdx.x) * nt) / gridDim.x);
    const int t_end = int((int64_t(blockIdx.x + 1) * nt) / gridDim.x);
    const int ntl = t_end - t_begin;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(su32(&bars->full[s]), 1);
            mbar_init(su32(&bars->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(su32(&bars->acc_full[b]), 1);
            mbar_init(su32(&bars->acc_empty[b]), 4);
        }
        mbar_init(su32(&bars->e_ready), kLanes);
        mbar_init(su32(&bars->drain), 1);
        bars->wc.flag = 0;
        bars->wc.limit_ns = t.wait_ns;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_wait();   // previous tokens and base rows may come from the kernel just before
    if (warp == 4) tc_alloc(su32(&bars->tmem_base), kCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    int done_steps = 0;   // epilogue: steps whose picks are written

    if (warp == 5) {
        // ------------------------------------------------------------ TMA producer, every step
        if (lane == 0) {
            const uint64_t keep = l2_evict_last();
            const int total = steps * ntl * kKB;
            int issued = 0;
            for (int i = 0; i < total; ++i) {
                const int s = i % kStages;
                if (i >= kStages && !mbar_wait(su32(&bars->empty[s]), ((i / kStages) - 1) & 1, abortp)) break;
                const int il = i % (ntl * kKB);   // k-block within the step
                const uint32_t bar = su32(&bars->full[s]);
                mbar_expect_tx(bar, kSlabB);
                tma_load_2d_hint(sB + s * kSlabB, &w2map, (il % kKB) * 64, (t_begin + il / kKB) * kTileV, bar, keep);
                ++issued;
            }
            if (abortp->flag)
                for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
                    mbar_drain(su32(&bars->full[i % kStages]), (i / kStages) & 1);
        }
        __syncwarp();
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA, every step
        if (lane == 0) {
            bool ok = true;
            for (int j = 0; j < steps && ok; ++j) {
                ok = mbar_wait(su32(&bars->e_ready), j & 1, abortp);   // the step's W1 rows are in E
                if (!ok) break;
                tc_fence_after();
                for (int tt = 0; tt < ntl && ok; ++tt) {
                    const int gt = j * ntl + tt, b = gt & 1;
                    if (gt >= 2) {
                        ok = mbar_wait(su32(&bars->acc_empty[b]), ((gt >> 1) - 1) & 1, abortp);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    for (int kb = 0; kb < kKB && ok; ++kb) {
                        const int i = gt * kKB + kb, s = i % kStages;
                        ok = mbar_wait(su32(&bars->full[s]), (i / kStages) & 1, abortp);
                        if (!ok) break;
                        tc_fence_after();
                        const uint64_t da = sdesc(sA + kb * kSlabB, 16, 1024);
                        const uint64_t db = sdesc(sB + s * kSlabB, 16, 1024);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            tc_mma_ss(tmem + uint32_t(b * kTileV), da + 2 * k, db + 2 * k, kIdesc,
                                      (kb | k) ? 1u : 0u);
                        tc_commit(su32(&bars->empty[s]));
                    }
                    if (ok) tc_commit(su32(&bars->acc_full[b]));
                }
            }
            tc_commit(su32(&bars->drain));
            mbar_drain(su32(&bars->drain), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue + W1 gather, every step
        const int L = 4 * lane + warp;   // the stream on TMEM lane 32*warp + lane
        const uint32_t tlane = tmem + (uint32_t(warp * 32) << 16);
        // this CTA's slice of stream tid's base row of step jj into L2 (rows do
        // not depend on the picks, so a step ahead; whole 16-byte units only)
        auto prefetch_base = [&](int jj) {
            if (tid < t.S && jj < steps) {
                const SegStream st = t.streams[tid];
                if (st.rows - 1 > jj) {
                    const int v_begin = t_begin * kTileV;
                    const int v_end = min(t_end * kTileV, vocab);
                    const uint32_t bytes = uint32_t(v_end - v_begin) * 2u & ~15u;
                    if (bytes) l2_prefetch_bulk(base + int64_t(st.row_offset - tid + jj) * base_stride + v_begin, bytes);
                }
            }
        };
        prefetch_base(0);
        // Every exit from this loop is taken by the four warps together: the
        // decision is thread 0's snapshot (bars->stop), written before a
        // barrier and read after it.
        for (int j = 0; j < steps; ++j) {
            // the previous step's picks are written (step barrier), then this step's tokens
            if (j > 0) {
                if (tid == 0) {
                    chain_wait(t.mk_sync, uint32_t(j), abortp);
                    bars->stop = abortp->flag ? 1 : 0;
                }
                epi_sync();
                if (bars->stop) break;
            }
            {
                const int s = tid;
                int tok = -1, row = -1;
                if (s < t.S) {
                    const SegStream st = t.streams[s];
                    if (st.rows - 1 > j) {
                        row = st.row_offset - s + j;
                        tok = j == 0 ? prev[s] : __ldcg(pick + row - 1);
                        if (tok < 0 || tok >= vocab) tok = -1;
                    }
                }
                bars->tok[tid] = tok;
                bars->row[tid] = row;
            }
            epi_sync();
            // E = the streams' W1 rows (every MMA of the step before has completed:
            // this warp group read each of its accumulators)
            for (int idx = tid; idx < kLanes * (TF_MK / 8); idx += kLanes) {
                const int Ls = idx >> 5, c = idx & 31, m = lane_of(Ls);
                const int tok = bars->tok[Ls];
                const uint16_t* src = tok >= 0 ? W1 + size_t(tok) * TF_MK + c * 8 : W1;
                cp_async16(sA + (c >> 3) * kSlabB + m * 128 + (((c & 7) ^ (m & 7)) << 4), src, tok >= 0);
            }
            asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
            fence_async_smem();
            mbar_arrive(su32(&bars->e_ready));
            prefetch_base(j + 1);

            const int my_tok = bars->tok[L];
            const int my_row = bars->row[L];
            const bool valid = my_tok >= 0;
            const bool wact = __any_sync(0xFFFFFFFFu, valid);
            const uint16_t* brow = base + (valid ? my_row : 0) * base_stride;
            float best = -INFINITY;
            int bid = 0x7FFFFFFF;
            uint32_t nf = 0;
            uint32_t cur[64], nxt[64];
            if (wact && ntl > 0) load_base_tile(brow, t_begin * kTileV, vocab, cur);
            bool ok = true;
            for (int tt = 0; tt < ntl; ++tt) {
                const int gt = j * ntl + tt, b = gt & 1;
                const int v0 = (t_begin + tt) * kTileV;
                if (wact && tt + 1 < ntl) load_base_tile(brow, v0 + kTileV, vocab, nxt);
                if (!mbar_wait_warp(su32(&bars->acc_full[b]), (gt >> 1) & 1, abortp)) {
                    ok = false;   // leaves the tile loop only: the step's barriers below are still met
                    break;
                }
                tc_fence_after();
                if (wact) {
                    // two pieces of 32 columns in flight: the next one loads while
                    // this one is scored
                    uint32_t ra[32], rb[32];
                    tc_ld_n<32>(tlane + uint32_t(b * kTileV), ra);
#pragma unroll
                    for (int p = 0; p < kTileV / 32; ++p) {
                        tc_wait_ld();
                        uint32_t(&r)[32] = (p & 1) ? rb : ra;
                        if (p + 1 < kTileV / 32)
                            tc_ld_n<32>(tlane + uint32_t(b * kTileV + 32 * (p + 1)), (p & 1) ? ra : rb);
                        const int v = v0 + 32 * p;
                        if (v < vocab && valid) {
                            const int n = vocab - v < 32 ? vocab - v : 32;
                            score_piece(r, cur + 16 * p, v, n, best, bid, nf);
                        }
                    }
                    tc_wait_ld();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(su32(&bars->acc_empty[b]));
#pragma unroll
                for (int k = 0; k < 64; ++k) cur[k] = nxt[k];
            }
            nf = (nf & 0x80008000u) ? 1u : 0u;
            if (valid && ok) {
                if (bid != 0x7FFFFFFF)
                    atomicMax(&t.mk_keys[L], (static_cast<unsigned long long>(ord_bf16(best)) << 32) |
                                                 static_cast<unsigned long long>(0xFFFFFFFFu - uint32_t(bid)));
                if (nf) atomicOr(&t.mk_flags[L], 1u);
            }
            __threadfence();
            epi_sync();
            if (tid == 0) {
                bars->stop = abortp->flag ? 1 : 0;
                bars->last = 0;
                if (!bars->stop) {
                    __threadfence();
                    bars->last = atomicAdd(t.mk_sync, 1u) == uint32_t(j + 1) * gridDim.x - 1;
                }
            }
            epi_sync();
            if (bars->stop) break;
            if (bars->last) {
                // the step's picks and flags, then its scratch back to zero
                __threadfence();
                if (bars->row[tid] >= 0) {
                    const unsigned long long key = atomicExch(&t.mk_keys[tid], 0ull);
                    const uint32_t fl = atomicExch(&t.mk_flags[tid], 0u);
                    int p = -1;
                    uint8_t f = 1;
                    if (bars->tok[tid] >= 0) {
                        if (fl) {
                            f = uint8_t(fl);
                        } else {
                            p = int(0xFFFFFFFFu - uint32_t(key & 0xFFFFFFFFull));
                            f = 0;
                        }
                    }
                    pick[bars->row[tid]] = p;
                    flag[bars->row[tid]] = f;
                }
                __threadfence();
                epi_sync();
                if (tid == 0) {   // open the next step
                    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(t.mk_sync + 1), "r"(uint32_t(j + 1))
                                 : "memory");
                }
            }
            done_steps = j + 1;
        }
        if (abortp->flag) {
            // give up: the other CTAs stop waiting; this stream's rows of the
            // steps not done are flagged
            atomicExch(t.mk_sync + 2, 1u);
            if (tid < t.S) {
                const SegStream st = t.streams[tid];
                for (int j = done_steps; j + 1 < st.rows; ++j) {
                    pick[st.row_offset - tid + j] = -1;
                    flag[st.row_offset - tid + j] = 2;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    if (tid == 0 && abortp->flag) atomicOr(t.status, uint32_t(TF_STATUS_MARKOV_TIMEOUT));
    if (warp == 4) {
        tc_fence_after();
        tc_dealloc(tmem, kCols);
    }
}


// ---- the whole chain with W2 held on chip (tables of at most 64 streams) --
//
// Streaming W2 (65.5 MB at a 128,000-token vocabulary) through every step
// makes a step cost one pass over it at the rate L2 delivers it to the SMs,
// which measured no better than HBM's. Most of W2 fits on chip across the
// 152 SMs instead: with at most 64 streams the step is computed transposed,
// D[v][s] = W2[v] . E[s] (MMA M = 128 vocabulary rows, N = 32 or 64 streams,
// K = 256), so that W2 is the A operand, which tcgen05 can read from tensor
// memory. Each CTA (one per SM) keeps the first three of its W2 tiles in
// tensor memory (128 columns each, written once at the start), the fourth in
// shared memory (loaded once), and streams the rest through a ring of 16 KB
// k-blocks every step. A step visits the first streamed tile first (its
// k-blocks arrive while the CTAs meet between steps), then the held tiles
// (while the ring refills), then the other streamed ones.
//
// Transposed, each TMEM lane holds one vocabulary row and each column one
// stream. The epilogue works lane-major: thread = lane = vocabulary row, and
// two groups of four warps split the streams (group g takes streams
// [g*N/2, (g+1)*N/2)). Per tile a thread rounds its dot products to bf16 two
// streams at a time, adds the base logits (staged per tile in shared memory
// by a producer warp of its own, in 16-byte asynchronous copies: stream s's
// 128 logits as one 256-byte row; W2's ring has another, so that it never
// waits behind these copies), and keeps per stream the largest score with its tile
// (packed bf16 compare and max, the tiles merged in vocabulary order, so a
// strict compare keeps the first) and a nonfinite bit. The argmax along the vocabulary is then taken once a
// step: a shuffle reduction over the warp's lanes of (ordered score, lowest
// row) keys, then over the four warps.
//
// Between steps the CTAs meet through the table's scratch, three generations
// deep: each CTA atomicMax-es its key per stream into one of eight keys per
// stream (CTA c into key c % 8, which keeps same-address atomics few), counts
// its arrival, and once the count shows every CTA, every CTA reads the eight
// keys and the flags and takes the picks itself, so no CTA has to publish
// them before the next step; CTA 0 writes the outputs and clears the
// generation two steps ahead. Before it arrives, a CTA asks L2 for the W1
// rows of its own best tokens, one of which is each stream's next token.
// Waits are bounded as in the other kernels; a CTA that gives up raises the
// launch's abort word, and CTA 0 marks the rows of the steps not done (flag
// bit 1).

constexpr int kTmTiles = 3;       // W2 tiles a CTA holds in tensor memory
constexpr int kSmTiles = 1;       // W2 tiles a CTA holds in shared memory
constexpr int kKeyGroups = 8;     // per-stream keys CTAs meet in (CTA c in key c % 8)
constexpr int kMaxDynSmem = 232448;
constexpr int kRingMax = 12;
constexpr int kBaseBufs = 3;      // tiles of base logits staged ahead
constexpr uint32_t kHoldCols = 512;
constexpr int kHoldEpi = 256;                     // epilogue threads: two groups of four warps
constexpr int kHoldMmaWarp = 8, kHoldTmaWarp = 9, kHoldBaseWarp = 10;
constexpr int kHoldThreads = kHoldEpi + 96;

struct HoldBars {
    uint64_t full[kRingMax];
    uint64_t empty[kRingMax];
    uint64_t bfull[kBaseBufs];   // a tile's base logits have landed (each producer lane's copies)
    uint64_t bempty[kBaseBufs];  // the 8 epilogue warps have read them
    uint64_t acc_full[2];
    uint64_t acc_empty[2];       // the 8 epilogue warps have read the accumulator
    uint64_t e_ready;            // E holds the step's W1 rows (the 256 epilogue threads)
    uint64_t tm_ready;           // the tensor-memory tiles are written (the 256 epilogue threads)
    uint64_t res_full;           // the shared-memory tile has landed
    uint64_t drain;
    uint32_t tmem_base;
    int32_t stop;                // epilogue thread 0's snapshot of the abort flag, read after a barrier
    WaitCtl wc;
    int32_t tok[64];             // the step's previous token of stream s, -1 if none or invalid
    int32_t row[64];             // the step's draft row of stream s, -1 if it has none
    uint32_t wkey[8][32];        // step end: each warp's best key per stream of its group (all ones: nonfinite)
};

template <int kN>
struct Hold {
    static constexpr int kS = kN / 2;                     // streams per epilogue group
    static constexpr int kEB = kKB * kN * 128;            // E: kN rows x 256, four k-blocks of kN x 128 B
    static constexpr int kBaseB = kN * kTileV * 2;        // one tile of base logits: [stream][128] bf16
    static constexpr int kResB = kSmTiles * kKB * kSlabB;
    static constexpr int kFixed = 1024 + kEB + kResB + kBaseBufs * kBaseB + int(sizeof(HoldBars));
    static constexpr int kRingFit = (kMaxDynSmem - kFixed) / kSlabB;
    static constexpr int kRing = kRingFit < kRingMax ? kRingFit : kRingMax;
    static constexpr int kSmem = kFixed + kRing * kSlabB;
    static constexpr uint32_t kAcc = kTmTiles * 128;      // tensor-memory column of accumulator 0
    // kind::f16, fp32 accumulate, A and B bf16 K-major, N = kN, M = 128
    static constexpr uint32_t kIdesc =
        (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(kN >> 3) << 17) | (uint32_t(128 >> 4) << 24);
    static_assert(kRing >= 4, "the ring holds at least one tile");
    static_assert(kAcc + 2 * kN <= kHoldCols, "tiles and accumulators fit tensor memory");
    static_assert(kS == 16 || kS == 32, "streams per group");
};

// tcgen05.mma with the accumulate flag as an immediate (0: overwrite D)
template <int ACC>
__device__ __forceinline__ void tc_mma_ss_acc(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
                 ::"r"(d), "l"(a), "l"(b), "r"(idesc), "n"(ACC) : "memory");
}
template <int ACC>
__device__ __forceinline__ void tc_mma_ts_acc(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc) {
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
                 ::"r"(d), "r"(a), "l"(b), "r"(idesc), "n"(ACC) : "memory");
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
// packed bf16 pair compare: each 16-bit half all ones where a > b (ordered; 0 for NaN)
__device__ __forceinline__ uint32_t gt_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("set.gt.u32.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

template <int kN>
__global__ void __launch_bounds__(kHoldThreads, 1)
markov_hold_kernel(SegTable t, int steps, const uint16_t* __restrict__ W1, const uint16_t* __restrict__ W2,
                   int vocab, const uint16_t* __restrict__ base, int64_t base_stride,
                   const int32_t* __restrict__ prev, int32_t* __restrict__ pick, uint8_t* __restrict__ flag,
                   const __grid_constant__ CUtensorMap w2map) {
    using C = Hold<kN>;
    constexpr int kS = C::kS;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = su32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    unsigned char* gbase = smem_raw + (sbase - raw);
    const uint32_t sE = sbase;
    const uint32_t sRes = sE + C::kEB;
    const uint32_t sBase = sRes + C::kResB;
    const uint32_t sRing = sBase + kBaseBufs * C::kBaseB;
    HoldBars* bars = reinterpret_cast<HoldBars*>(gbase + (sRing - sbase) + C::kRing * kSlabB);
    volatile WaitCtl* abortp = &bars->wc;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nt = (vocab + kTileV - 1) / kTileV;
    const int t_begin = int((int64_t(blockIdx.x) * nt) / gridDim.x);
    const int t_end = int((int64_t(blockIdx.x + 1) * nt) / gridDim.x);
    const int ntl = t_end - t_begin;
    const int nT = ntl < kTmTiles ? ntl : kTmTiles;                      // [0, nT) in tensor memory
    const int nR = ntl < kTmTiles + kSmTiles ? ntl : kTmTiles + kSmTiles;   // [nT, nR) in shared memory
    const int ns = ntl - nR;                                             // [nR, ntl) streamed every step
    // the i-th tile of a step: the first streamed tile (its k-blocks already in
    // the ring when the step starts), the held tiles, then the other streamed ones,
    // so that the ring refills while the held tiles run
    auto order = [&](int i) { return ns == 0 ? i : (i == 0 ? nR : (i <= nR ? i - 1 : i)); };
    uint32_t* sync = t.mk_sync;                                          // [0] arrivals, [2] abort
    uint32_t* gflags = sync + 64;                                        // [3][64]
    unsigned long long* gkeys = reinterpret_cast<unsigned long long*>(sync + 256);   // [3][kKeyGroups][64]

    if (tid == 0) {
        for (int s = 0; s < C::kRing; ++s) {
            mbar_init(su32(&bars->full[s]), 1);
            mbar_init(su32(&bars->empty[s]), 1);
        }
        for (int q = 0; q < kBaseBufs; ++q) {
            mbar_init(su32(&bars->bfull[q]), 32);   // the producer's 32 lanes, as their copies land
            mbar_init(su32(&bars->bempty[q]), 8);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(su32(&bars->acc_full[b]), 1);
            mbar_init(su32(&bars->acc_empty[b]), 8);
        }
        mbar_init(su32(&bars->e_ready), kHoldEpi);
        mbar_init(su32(&bars->tm_ready), kHoldEpi);
        mbar_init(su32(&bars->res_full), 1);
        mbar_init(su32(&bars->drain), 1);
        bars->wc.flag = 0;
        bars->wc.limit_ns = t.wait_ns;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_wait();
    if (warp == kHoldMmaWarp) tc_alloc(su32(&bars->tmem_base), kHoldCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == kHoldTmaWarp) {
        // ------------------------------------------------------------ W2 producer (lane 0)
        // the shared-memory tile once, the streamed tiles' k-blocks through the
        // ring every step (a slot frees when the MMAs reading it complete, so
        // the ring refills across step boundaries). Bounded: no progress for
        // the wait limit (or another thread's give-up) ends it.
        if (lane == 0) {
            const uint64_t keep = l2_evict_last();
            {   // the tensor-memory tiles' rows (contiguous in W2) into L2 for the epilogue's loads
                const int64_t r0 = int64_t(t_begin) * kTileV;
                const int64_t r1 = min(int64_t(t_begin + nT) * kTileV, int64_t(vocab));
                if (r1 > r0) l2_prefetch_bulk(W2 + r0 * TF_MK, uint32_t((r1 - r0) * TF_MK * 2));
            }
            if (nR > nT) {
                mbar_expect_tx(su32(&bars->res_full), uint32_t(C::kResB));
                for (int kb = 0; kb < kKB; ++kb)
                    tma_load_2d_hint(sRes + kb * kSlabB, &w2map, kb * 64, (t_begin + nT) * kTileV,
                                     su32(&bars->res_full), keep);
            }
            const int per_step_r = ns * kKB, total_r = steps * per_step_r;
            int gr = 0;
            bool ok = true;
            unsigned long long idle0 = gtime();
            while (ok && gr < total_r) {
                const int s = gr % C::kRing;
                if (gr < C::kRing || mbar_test(su32(&bars->empty[s]), ((gr / C::kRing) - 1) & 1)) {
                    const int il = gr % per_step_r;
                    const uint32_t bar = su32(&bars->full[s]);
                    mbar_expect_tx(bar, kSlabB);
                    tma_load_2d_hint(sRing + s * kSlabB, &w2map, (il % kKB) * 64,
                                     (t_begin + nR + il / kKB) * kTileV, bar, keep);
                    ++gr;
                    idle0 = gtime();
                } else if (abortp->flag) {
                    ok = false;
                } else if (gtime() - idle0 > abortp->limit_ns) {
                    abortp->flag = 1;
                    ok = false;
                } else {
                    __nanosleep(20);
                }
            }
            if (!ok) {
                // let the copies in flight land before the CTA exits (bounded waits)
                for (int i = gr > C::kRing ? gr - C::kRing : 0; i < gr; ++i)
                    mbar_drain(su32(&bars->full[i % C::kRing]), (i / C::kRing) & 1);
                if (nR > nT) mbar_drain(su32(&bars->res_full), 0);
            }
        }
        __syncwarp();
    } else if (warp == kHoldBaseWarp) {
        // ------------------------------------------------------------ base logits producer
        // each tile's base logits, in step order (a buffer frees when the
        // epilogue has read it), lane l copying the rows of streams l and
        // l + 32; a warp of its own, so that W2's ring never waits behind
        // these copies. Bounded like the W2 producer.
        int rows_s[2] = {0, 0}, off_s[2] = {0, 0};   // streams lane and lane + 32
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int s = lane + 32 * h;
            if (s < kN && s < t.S) {
                const SegStream st = t.streams[s];
                rows_s[h] = st.rows;
                off_s[h] = st.row_offset - s;
            }
        }
        const int total_b = steps * ntl;
        int gb = 0;
        bool ok = true;
        unsigned long long idle0 = gtime();
        while (ok && gb < total_b) {
            const int q = gb % kBaseBufs;
            bool free_q = gb < kBaseBufs;
            if (!free_q && lane == 0) free_q = mbar_test(su32(&bars->bempty[q]), ((gb / kBaseBufs) - 1) & 1);
            if (__shfl_sync(0xFFFFFFFFu, free_q ? 1 : 0, 0)) {
                // 16-byte asynchronous copies through the load path (many small bulk
                // copies would queue on the SM's one TMA unit, ahead of W2), through
                // L1 so that the two halves of each 32-byte sector are fetched from L2 once
                const int j = gb / ntl, i = gb - j * ntl;
                const int v0 = (t_begin + order(i)) * kTileV;
                // 128 logits, or the vocabulary's tail rounded up to 16 bytes (within
                // the row: the stride is a multiple of 8 elements and at least the vocabulary)
                const int nv = vocab - v0 < kTileV ? vocab - v0 : kTileV;
                const int nchunk = (nv + 7) >> 3;
                const uint32_t dst = sBase + uint32_t(q * C::kBaseB);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (rows_s[h] - 1 > j) {
                        const uint16_t* src = base + int64_t(off_s[h] + j) * base_stride + v0;
                        const uint32_t d = dst + uint32_t((lane + 32 * h) * 256);
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            if (c < nchunk)
                                asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(d + c * 16),
                                             "l"(src + c * 8) : "memory");
                    }
                }
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(su32(&bars->bfull[q]))
                             : "memory");
                ++gb;
                idle0 = gtime();
            } else {
                bool give_up = false;
                if (lane == 0) {
                    if (abortp->flag) {
                        give_up = true;
                    } else if (gtime() - idle0 > abortp->limit_ns) {
                        abortp->flag = 1;
                        give_up = true;
                    }
                }
                ok = !__shfl_sync(0xFFFFFFFFu, give_up ? 1 : 0, 0);
                __nanosleep(20);
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");   // every lane's base copies have landed
        __syncwarp();
    } else if (warp == kHoldMmaWarp) {
        // ------------------------------------------------------------ MMA
        // One thread issues every MMA, so the issue path is kept short:
        // descriptors are formed once and advanced by constants (a shared-memory
        // descriptor's address field counts 16-byte units), every K loop is
        // unrolled, and the accumulate flag is an immediate.
        if (lane == 0) {
            const uint64_t dE0 = sdesc(sE, 16, 1024);
            const uint64_t dRes0 = sdesc(sRes, 16, 1024);
            const uint64_t dRing0 = sdesc(sRing, 16, 1024);
            constexpr uint32_t kEkb = uint32_t(kN * 128) >> 4;   // E's k-block stride, 16-byte units
            constexpr uint32_t kSlab16 = uint32_t(kSlabB) >> 4;
            bool ok = true, tm_seen = false, res_seen = false;
            int si = 0;   // streamed k-blocks consumed
            for (int j = 0; j < steps && ok; ++j) {
                ok = mbar_wait(su32(&bars->e_ready), j & 1, abortp);
                if (!ok) break;
                tc_fence_after();
                for (int i = 0; i < ntl && ok; ++i) {
                    const int gt = j * ntl + i, b = gt & 1;
                    if (gt >= 2) {
                        ok = mbar_wait(su32(&bars->acc_empty[b]), ((gt >> 1) - 1) & 1, abortp);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    const int lt = order(i);
                    const uint32_t d = tmem + C::kAcc + uint32_t(b * kN);
                    if (lt < nT) {
                        if (!tm_seen) {
                            ok = mbar_wait(su32(&bars->tm_ready), 0, abortp);
                            tm_seen = true;
                            if (!ok) break;
                            tc_fence_after();
                        }
                        const uint32_t a = tmem + uint32_t(lt * 128);   // A: 8 tensor-memory columns per 16 of K
#pragma unroll
                        for (int k = 0; k < TF_MK / 16; ++k) {
                            const uint64_t db = dE0 + uint64_t((k >> 2) * kEkb + 2 * (k & 3));
                            if (k == 0)
                                tc_mma_ts_acc<0>(d, a, db, C::kIdesc);
                            else
                                tc_mma_ts_acc<1>(d, a + uint32_t(8 * k), db, C::kIdesc);
                        }
                    } else if (lt < nR) {
                        if (!res_seen) {
                            ok = mbar_wait(su32(&bars->res_full), 0, abortp);
                            res_seen = true;
                            if (!ok) break;
                            tc_fence_after();
                        }
                        const uint64_t da0 = dRes0 + uint64_t(uint32_t(lt - nT) * kKB * kSlab16);
#pragma unroll
                        for (int k = 0; k < TF_MK / 16; ++k) {
                            const uint64_t da = da0 + uint64_t((k >> 2) * kSlab16 + 2 * (k & 3));
                            const uint64_t db = dE0 + uint64_t((k >> 2) * kEkb + 2 * (k & 3));
                            if (k == 0)
                                tc_mma_ss_acc<0>(d, da, db, C::kIdesc);
                            else
                                tc_mma_ss_acc<1>(d, da, db, C::kIdesc);
                        }
                    } else {
#pragma unroll
                        for (int kb = 0; kb < kKB; ++kb) {
                            const int s = si % C::kRing;
                            if (!ok || !mbar_wait(su32(&bars->full[s]), (si / C::kRing) & 1, abortp)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint64_t da0 = dRing0 + uint64_t(uint32_t(s) * kSlab16);
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const uint64_t db = dE0 + uint64_t(kb * kEkb + 2 * k);
                                if (kb == 0 && k == 0)
                                    tc_mma_ss_acc<0>(d, da0, db, C::kIdesc);
                                else
                                    tc_mma_ss_acc<1>(d, da0 + uint64_t(2 * k), db, C::kIdesc);
                            }
                            tc_commit(su32(&bars->empty[s]));
                            ++si;
                        }
                    }
                    if (ok) tc_commit(su32(&bars->acc_full[b]));
                }
            }
            tc_commit(su32(&bars->drain));
            mbar_drain(su32(&bars->drain), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue: two groups of 128 threads
        // thread et = TMEM lane = row et of every tile; group wg takes streams [wg*kS, wg*kS + kS)
        const int wg = tid >> 7, et = tid & 127;
        const uint32_t tlane = tmem + (uint32_t((warp & 3) * 32) << 16);
        auto all_sync = [&]() { asm volatile("bar.sync 1, 256;" ::: "memory"); };
        auto prefetch_base = [&](int jj) {   // this CTA's slice of stream tid's base row of step jj into L2
            if (tid < t.S && jj < steps) {
                const SegStream st = t.streams[tid];
                if (st.rows - 1 > jj) {
                    const int v_begin = t_begin * kTileV;
                    const int v_end = min(t_end * kTileV, vocab);
                    const uint32_t bytes = uint32_t(v_end - v_begin) * 2u & ~15u;
                    if (bytes)
                        l2_prefetch_bulk(base + int64_t(st.row_offset - tid + jj) * base_stride + v_begin, bytes);
                }
            }
        };
        if (tid < 64) {
            int tok = -1, row = -1;
            if (tid < t.S) {
                const SegStream st = t.streams[tid];
                if (st.rows > 1) {
                    row = st.row_offset - tid;
                    tok = prev[tid];
                    if (tok < 0 || tok >= vocab) tok = -1;
                }
            }
            bars->tok[tid] = tok;
            bars->row[tid] = row;
        }
        prefetch_base(0);
        all_sync();
        int done_steps = 0;
        for (int j = 0; j < steps; ++j) {
            // E = the step's W1 rows (zero rows for streams without a token)
            for (int idx = tid; idx < kN * (TF_MK / 8); idx += kHoldEpi) {
                const int m = idx >> 5, c = idx & 31;
                const int tok = bars->tok[m];
                const uint16_t* src = tok >= 0 ? W1 + size_t(tok) * TF_MK + c * 8 : W1;
                cp_async16(sE + (c >> 3) * (kN * 128) + m * 128 + (((c & 7) ^ (m & 7)) << 4), src, tok >= 0);
            }
            asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
            fence_async_smem();
            mbar_arrive(su32(&bars->e_ready));
            if (j == 0) {
                // the held tensor-memory tiles, group wg taking tiles wg, wg + 2, ...: lane et takes
                // W2 row (tile start + et), 512 bytes, 64 columns at a time (zeros past the vocabulary)
                for (int r = wg; r < nT; r += 2) {
                    const int64_t vrow = int64_t(t_begin + r) * kTileV + et;
                    const bool in = vrow < vocab;
                    const uint4* src = reinterpret_cast<const uint4*>(W2 + (in ? vrow : 0) * TF_MK);
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        uint32_t w0[32], w1[32];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const uint4 x = in ? __ldg(src + 16 * q + u) : make_uint4(0, 0, 0, 0);
                            const uint4 y = in ? __ldg(src + 16 * q + 8 + u) : make_uint4(0, 0, 0, 0);
                            w0[4 * u] = x.x; w0[4 * u + 1] = x.y; w0[4 * u + 2] = x.z; w0[4 * u + 3] = x.w;
                            w1[4 * u] = y.x; w1[4 * u + 1] = y.y; w1[4 * u + 2] = y.z; w1[4 * u + 3] = y.w;
                        }
                        tc_st_n<32>(tlane + uint32_t(r * 128 + 64 * q), w0);
                        tc_st_n<32>(tlane + uint32_t(r * 128 + 64 * q + 32), w1);
                    }
                }
                tc_wait_st();
                tc_fence_before();
                mbar_arrive(su32(&bars->tm_ready));
            }
            prefetch_base(j + 1);

            // per stream pair of the group: the largest score so far (bf16 pair), the
            // tile holding each, and nonfinite bits (bit 15 / 31)
            // (the first streamed tile, visited first, is held aside as scores and
            // merged after the held tiles, so that the running maximum sees the tiles
            // in vocabulary order)
            // btile: the tile of each best, two 16-bit halves like the scores
            uint32_t best[kS / 2], nfa[kS / 2], early[kS / 2], btile[kS / 2];
#pragma unroll
            for (int p = 0; p < kS / 2; ++p) {
                best[p] = 0xFF80FF80u;   // -inf, -inf
                early[p] = 0xFF80FF80u;
                nfa[p] = 0u;
                btile[p] = 0u;
            }
            bool ok = true;
            for (int i = 0; i < ntl; ++i) {
                const int gt = j * ntl + i, b = gt & 1, q = gt % kBaseBufs;
                // (a warp that gave up still meets every barrier of the step, doing no work)
                if (ok && mbar_wait_warp(su32(&bars->acc_full[b]), (gt >> 1) & 1, abortp)) {
                    tc_fence_after();
                    uint32_t a[kS];
                    tc_ld_n<kS>(tlane + C::kAcc + uint32_t(b * kN + wg * kS), a);
                    tc_wait_ld();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(su32(&bars->acc_empty[b]));
                    if (mbar_wait_warp(su32(&bars->bfull[q]), (gt / kBaseBufs) & 1, abortp)) {
                        const int lt = order(i);
                        const uint32_t bb = sBase + uint32_t(q * C::kBaseB + wg * kS * 256 + et * 2);
                        if ((t_begin + lt) * kTileV + et < vocab) {
                            const bool hold = ns > 0 && i == 0;
                            const uint32_t ltp = uint32_t(lt) * 0x00010001u;
#pragma unroll
                            for (int p = 0; p < kS / 2; ++p) {
                                const uint32_t lo = lds16(bb + uint32_t((2 * p) * 256));
                                const uint32_t hi = lds16(bb + uint32_t((2 * p + 1) * 256));
                                const uint32_t sc = add_bf16x2(
                                    cvt_bf16x2(__uint_as_float(a[2 * p + 1]), __uint_as_float(a[2 * p])), lo | (hi << 16));
                                nfa[p] |= (sc & 0x7F807F80u) + 0x00800080u;
                                if (hold) {
                                    early[p] = sc;
                                } else {
                                    const uint32_t g = gt_bf16x2(sc, best[p]);
                                    best[p] = max_bf16x2(best[p], sc);
                                    btile[p] = (btile[p] & ~g) | (ltp & g);
                                }
                            }
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(su32(&bars->bempty[q]));
                    } else {
                        ok = false;
                    }
                } else {
                    ok = false;
                }
                if (ns > 0 && i == nR) {   // the held tiles are in: the first streamed tile (tile nR) next
#pragma unroll
                    for (int p = 0; p < kS / 2; ++p) {
                        const uint32_t g = gt_bf16x2(early[p], best[p]);
                        best[p] = max_bf16x2(best[p], early[p]);
                        btile[p] = (btile[p] & ~g) | ((uint32_t(nR) * 0x00010001u) & g);
                    }
                }
            }
            // ---- the argmax along the vocabulary: warp, then the group's four warps
            // key = (ordered score << 16) | (0xFFFF - row within this CTA's range): the
            // largest key is the largest score at the lowest row; a nonfinite score
            // anywhere makes the stream's key all ones (above every score's)
            uint32_t key[kS];
#pragma unroll
            for (int p = 0; p < kS / 2; ++p) {
                const float lo = bf_lo(best[p]), hi = bf_hi(best[p]);
                key[2 * p] = (nfa[p] & 0x8000u)
                                 ? 0xFFFFFFFFu
                                 : (ord_bf16(lo) << 16) | (0xFFFFu - ((btile[p] & 0xFFFFu) * kTileV + uint32_t(et)));
                key[2 * p + 1] = (nfa[p] & 0x80000000u)
                                     ? 0xFFFFFFFFu
                                     : (ord_bf16(hi) << 16) | (0xFFFFu - ((btile[p] >> 16) * kTileV + uint32_t(et)));
            }
            // rows past the vocabulary never scored: their best stays -inf (key below any score's)
            // reduce-scatter: after the pass with offset o, lane l keeps the streams whose bit o is l's
#pragma unroll
            for (int o = kS / 2; o >= 1; o >>= 1) {
                const bool upper = (lane & o) != 0;
#pragma unroll
                for (int s = 0; s < o; ++s) {
                    const uint32_t send = upper ? key[s] : key[s + o];
                    const uint32_t keep = upper ? key[s + o] : key[s];
                    key[s] = max(keep, __shfl_xor_sync(0xFFFFFFFFu, send, o));
                }
            }
            if constexpr (kS == 16)   // lanes l and l ^ 16 hold the same stream: fold them
                key[0] = max(key[0], __shfl_xor_sync(0xFFFFFFFFu, key[0], 16));
            // lane l now holds stream l % kS of the group
            if (lane < kS) bars->wkey[warp][lane] = key[0];
            all_sync();
            const int b3 = j % 3;
            if (tid < kN && bars->tok[tid] >= 0) {
                const int g = tid / kS, sl = tid % kS;
                uint32_t k = 0;
#pragma unroll
                for (int w = 0; w < 4; ++w) k = max(k, bars->wkey[4 * g + w][sl]);
                // (a thread whose wait gave up has raised the abort flag: this CTA then
                // does not arrive, and the launch ends without these keys being read)
                if (k == 0xFFFFFFFFu) {
                    atomicOr(&gflags[b3 * 64 + tid], 1u);
                } else if (k >> 16) {
                    const uint32_t bidv = uint32_t(t_begin * kTileV) + (0xFFFFu - (k & 0xFFFFu));
                    const unsigned long long key64 =
                        (static_cast<unsigned long long>(k >> 16) << 32) | static_cast<unsigned long long>(0xFFFFFFFFu - bidv);
                    atomicMax(&gkeys[(b3 * kKeyGroups + int(blockIdx.x) % kKeyGroups) * 64 + tid], key64);
                    l2_prefetch_bulk(W1 + size_t(bidv) * TF_MK, TF_MK * 2);   // a candidate next token's W1 row
                }
            }
            if (blockIdx.x == 0) {   // clear the generation two steps ahead (read by every CTA before this step)
                const int bn = (j + 1) % 3;
                for (int idx = tid; idx < kKeyGroups * 64; idx += kHoldEpi) gkeys[bn * kKeyGroups * 64 + idx] = 0ull;
                if (tid < 64) gflags[bn * 64 + tid] = 0u;
            }
            __threadfence();
            all_sync();
            if (tid == 0) {
                if (!abortp->flag) {   // every wait of this CTA's step succeeded
                    atomicAdd(sync, 1u);
                    // every CTA has arrived (bounded: gives up on the wait limit or another CTA's abort)
                    const uint32_t target = uint32_t(j + 1) * gridDim.x;
                    const unsigned long long t0 = gtime(), limit = abortp->limit_ns;
                    for (;;) {
                        uint32_t g;
                        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(g) : "l"(sync) : "memory");
                        if (g >= target) break;
                        if (abortp->flag || *reinterpret_cast<const volatile uint32_t*>(sync + 2) ||
                            gtime() - t0 > limit) {
                            abortp->flag = 1;
                            break;
                        }
                        __nanosleep(32);
                    }
                }
                bars->stop = abortp->flag ? 1 : 0;
            }
            all_sync();
            if (bars->stop) break;
            // the step's picks, taken by every CTA; CTA 0 writes them out
            if (tid < 64) {
                const int row = bars->row[tid], tok = bars->tok[tid];
                int p = -1;
                uint8_t f = 1;
                if (row >= 0 && tok >= 0) {
                    // the flag word and the eight key groups in one round trip
                    const uint32_t fl = __ldcg(&gflags[b3 * 64 + tid]);
                    unsigned long long kg[kKeyGroups];
#pragma unroll
                    for (int g = 0; g < kKeyGroups; ++g) kg[g] = __ldcg(&gkeys[(b3 * kKeyGroups + g) * 64 + tid]);
                    if (fl) {
                        f = uint8_t(fl);
                    } else {
                        unsigned long long k = 0;
#pragma unroll
                        for (int g = 0; g < kKeyGroups; ++g) k = max(k, kg[g]);
                        p = int(0xFFFFFFFFu - uint32_t(k & 0xFFFFFFFFull));
                        f = 0;
                    }
                }
                if (blockIdx.x == 0 && row >= 0) {
                    pick[row] = p;
                    flag[row] = f;
                }
                int ntok = -1, nrow = -1;
                if (tid < t.S) {
                    const SegStream st = t.streams[tid];
                    if (st.rows - 1 > j + 1) {
                        nrow = st.row_offset - tid + j + 1;
                        ntok = (p >= 0 && p < vocab) ? p : -1;
                    }
                }
                bars->tok[tid] = ntok;
                bars->row[tid] = nrow;
            }
            done_steps = j + 1;
            all_sync();
        }
        if (abortp->flag || done_steps < steps) {
            abortp->flag = 1;
            atomicExch(sync + 2, 1u);   // the other CTAs stop waiting
            if (blockIdx.x == 0 && tid < t.S) {   // the rows of the steps not done
                const SegStream st = t.streams[tid];
                for (int j = done_steps; j + 1 < st.rows; ++j) {
                    pick[st.row_offset - tid + j] = -1;
                    flag[st.row_offset - tid + j] = 2;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    if (tid == 0 && abortp->flag) atomicOr(t.status, uint32_t(TF_STATUS_MARKOV_TIMEOUT));
    if (warp == kHoldMmaWarp) {
        tc_fence_after();
        tc_dealloc(tmem, kHoldCols);
    }
}

}  // namespace
}  // namespace tf

extern "C" int tf_markov_chain(const tf_segments* seg, const void* W1, const void* W2, int vocab, const void* base,
                               int64_t base_stride, const int32_t* prev, int32_t* pick, uint8_t* flag,
                               tf_cuda_stream stream) {
    using namespace tf;
    if (!W1 || !W2 || !base || !prev || !pick || !flag || vocab < 1) return TF_EINVAL;
    if (vocab > (1 << 24)) return TF_ERANGE;
    if (!aligned16(W1) || !aligned16(W2) || !aligned16(base) || base_stride < vocab || base_stride % 8 != 0)
        return TF_EINVAL;
    if (!seg || seg->prompt) return TF_EINVAL;
    if (seg->dev.S == 0 || seg->dev.R == seg->dev.S) return TF_OK;   // no window holds a draft
    SegTable t = seg->dev;
    t.wait_ns = wait_limit_ns();
    cudaError_t e = cudaFuncSetAttribute(markov_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e);
    CUtensorMap map;
    if (!encode_w2_map(&map, W2, vocab)) return cuda_fail(cudaErrorInvalidValue);
    const int nt = (vocab + kTileV - 1) / kTileV;
    const int gx = nt < sm_count() ? nt : sm_count();
    const dim3 grid(gx, (t.S + kLanes - 1) / kLanes);
    const uint16_t* w1 = static_cast<const uint16_t*>(W1);
    const uint16_t* b = static_cast<const uint16_t*>(base);
    const char* path = std::getenv("TF_MARKOV_PATH");
    const bool per_step = (path && std::strcmp(path, "step") == 0) || t.S > kLanes;
    const bool streamed = path && std::strcmp(path, "chain") == 0;
    // the held form keys a row within a CTA's range in 16 bits: at most 511 tiles a CTA
    if (!per_step && !streamed && t.S <= 64 && (nt + gx - 1) / gx <= 511) {
        // W2 held on chip, the whole chain in one cooperative launch
        auto* kern = t.S <= 32 ? markov_hold_kernel<32> : markov_hold_kernel<64>;
        const int smem = t.S <= 32 ? Hold<32>::kSmem : Hold<64>::kSmem;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return cuda_fail(e);
        e = cudaMemsetAsync(t.mk_sync, 0, kMkSyncBytes, stream);   // arrivals, abort word, keys and flags
        if (e != cudaSuccess) return cuda_fail(e);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(gx);
        cfg.blockDim = dim3(kHoldThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, t, t.max_rows - 1, w1, static_cast<const uint16_t*>(W2), vocab, b,
                               base_stride, prev, pick, flag, map);
        if (e != cudaSuccess) return cuda_fail(e);
        return launch_status();
    }
    if (!per_step) {
        // the whole chain in one cooperative launch (every CTA resident: one per SM)
        e = cudaFuncSetAttribute(markov_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kChainSmemBytes);
        if (e != cudaSuccess) return cuda_fail(e);
        e = cudaMemsetAsync(t.mk_sync, 0, 4 * sizeof(uint32_t), stream);   // the step barrier starts at zero
        if (e != cudaSuccess) return cuda_fail(e);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(gx);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kChainSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, markov_chain_kernel, t, t.max_rows - 1, w1, vocab, b, base_stride, prev, pick,
                               flag, map);
        if (e != cudaSuccess) return cuda_fail(e);
        return launch_status();
    }
    for (int j = 0; j + 1 < t.max_rows; ++j) {
        const int rc = launch_pdl(markov_step_kernel, grid, dim3(kThreads), kSmemBytes, stream, t, j, w1, vocab, b,
                                  base_stride, prev, pick, flag, map);
        if (rc != TF_OK) return rc;
    }
    return TF_OK;
}
