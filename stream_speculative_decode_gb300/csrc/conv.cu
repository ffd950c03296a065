// a1: LFM2 gated short conv over every row of every stream, one launch a layer.
//
// PR #1377 "LFM2: shared-round decode", commit "a shared round runs each
// layer's conv and attention once over all its streams": one launch a layer
// over every row from the segment table, each row's arithmetic that of the
// per-stream conv; streams longer than 8 rows are folded into 8-row tiles.
//
// Work split: a CTA owns one 8-row tile of one stream and 256 channels; its
// 128 threads are 32 channel groups (8 consecutive channels, 16-byte loads of
// B, C, x and the 3 taps) x 4 row slots, slot k taking the tile's rows k and
// k + 4 (128-thread CTAs, up to eight an SM: the next layer's CTAs find free
// slots sooner than with 256-thread ones, a 1,024-row layer 5.43 -> 5.36 us
// back to back). A table of few tiles of two rows or more on average takes
// one row per thread instead (16 groups x 8 slots, 128 channels a CTA: twice
// the CTAs); the arithmetic of a row is the same either way. Every thread loads its rows at once, gates them (bx = B*x) into
// shared memory, and after one barrier convolves each row with the two
// entries before it, so the rows of a tile run in parallel rather than one
// after the other. The two entries before a tile come from the conv state
// (first tile) or are recomputed from the input rows (later tiles), so tiles
// are independent. Only the first tile of a stream reads the state (rows 0
// and 1, before the barrier) and writes the new state (after it), so the
// in-place update needs no ordering between CTAs.
//
// HBM bound: per row 6144*2 B read + 2048*4 B written (+ state/history).
#include "tf_internal.cuh"

namespace tf {
namespace {

constexpr int kChan = 8;                        // channels per group
constexpr int kThreads = 128;
// The split of a CTA's 128 threads: RPT rows of the tile per thread, so
// 8 / RPT row slots (slot k takes rows k, k + 8/RPT, ...) and 128 * RPT / 8
// channel groups of 8 channels.
template <int RPT>
struct Split {
    static constexpr int kSlots = kConvTileRows / RPT;
    static constexpr int kGroups = kThreads / kSlots;
    static constexpr int kChanPerCta = kGroups * kChan;   // 256 (RPT 2) or 128 (RPT 1)
};

__device__ __forceinline__ void unpack8(const uint4& v, float f[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        f[2 * k] = __uint_as_float(w[k] << 16);
        f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}

// bx = bf16(B * x), round to nearest even: the fp32 product of two bf16 values
// is exact, so this is the single rounding of the gate.
__device__ __forceinline__ uint4 gate8(const uint4& b, const uint4& x) {
    float fb[8], fx[8];
    unpack8(b, fb);
    unpack8(x, fx);
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 p = __floats2bfloat162_rn(fb[2 * k] * fx[2 * k], fb[2 * k + 1] * fx[2 * k + 1]);
        o[k] = *reinterpret_cast<uint32_t*>(&p);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// bf16 element e (0..23) of the three packed tap vectors, as fp32
__device__ __forceinline__ float tap(const uint4 (&w)[3], int e) {
    const uint4& v = w[e >> 3];
    const int k = e & 7;
    const uint32_t word = (k >> 1) == 0 ? v.x : (k >> 1) == 1 ? v.y : (k >> 1) == 2 ? v.z : v.w;
    return __uint_as_float((k & 1) ? (word & 0xFFFF0000u) : (word << 16));
}

// y = C * (w0*e0 + w1*e1 + w2*bx) for 8 channels (entries oldest first), fp32
__device__ __forceinline__ void conv8(const uint4 (&w)[3], const uint4& e0, const uint4& e1, const uint4& bx,
                                      const uint4& cg, float o[8]) {
    float f0[8], f1[8], f2[8], fc[8];
    unpack8(e0, f0);
    unpack8(e1, f1);
    unpack8(bx, f2);
    unpack8(cg, fc);
#pragma unroll
    for (int k = 0; k < 8; ++k) {   // taps of channel k: elements 3k, 3k+1, 3k+2
        float conv = tap(w, 3 * k) * f0[k];
        conv = fmaf(tap(w, 3 * k + 1), f1[k], conv);
        conv = fmaf(tap(w, 3 * k + 2), f2[k], conv);
        o[k] = fc[k] * conv;
    }
}

template <int RPT>
__global__ void __launch_bounds__(kThreads, 8)
conv_rows_kernel(SegTable t, int layer, const uint16_t* __restrict__ bcx,
                 const uint16_t* __restrict__ w, float* __restrict__ y) {
    constexpr int kSlots = Split<RPT>::kSlots, kGroups = Split<RPT>::kGroups;
    constexpr int kChanPerCta = Split<RPT>::kChanPerCta;
    __shared__ uint4 sbx[kConvTileRows][kGroups];   // the tile's gated entries (4 or 2 KB)
    const ConvTile tile = t.tiles[blockIdx.x];
    const SegStream st = t.streams[tile.stream];
    const int grp = threadIdx.x % kGroups, slot = threadIdx.x / kGroups;
    const int c = blockIdx.y * kChanPerCta + grp * kChan;
    const size_t sl = size_t(layer) * t.S + tile.stream;
    uint16_t* state = static_cast<uint16_t*>(t.conv_state[sl]);
    uint16_t* hist = t.has_hist ? static_cast<uint16_t*>(t.conv_hist[sl]) : nullptr;
    const int n = tile.nrows;
    const int row_base = st.row_offset + tile.row0;
    const bool first = tile.row0 == 0;
    {
        // this thread's input rows into L2 while the previous kernel
        // finishes (a non-binding hint: L2 is the point of coherence, so a line the
        // previous kernel still writes is read after the wait as written)
#pragma unroll
        for (int k = 0; k < RPT; ++k) {
            const int j = slot + k * kSlots;
            if (j < n) {
                const uint16_t* row = bcx + size_t(row_base + j) * TF_CIN + c;
                asm volatile("prefetch.global.L2 [%0];" ::"l"(row));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(row + TF_H));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(row + 2 * TF_H));
            }
        }
    }
    pdl_wait();   // the table above; the data below may come from the previous kernel

    // this thread's rows slot, slot + kSlots, ... (loads issued before any arithmetic)
    uint4 B[RPT], C[RPT], X[RPT];
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        const int j = slot + k * kSlots;
        if (j < n) {
            const uint16_t* row = bcx + size_t(row_base + j) * TF_CIN + c;
            B[k] = __ldg(reinterpret_cast<const uint4*>(row));
            C[k] = __ldg(reinterpret_cast<const uint4*>(row + TF_H));
            X[k] = __ldg(reinterpret_cast<const uint4*>(row + 2 * TF_H));
        }
    }
    uint4 wv[3];   // taps of channels c..c+7: 24 bf16, element (channel j, tap k) at 3*j+k
    {
        const uint4* wp = reinterpret_cast<const uint4*>(w + size_t(c) * 3);
        wv[0] = __ldg(wp + 0);
        wv[1] = __ldg(wp + 1);
        wv[2] = __ldg(wp + 2);
    }
    // the two entries before the tile (rows 0 and 1 use them): the old state
    // for the first tile, else recomputed from the two input rows before it
    uint4 pm2 = make_uint4(0, 0, 0, 0), pm1 = make_uint4(0, 0, 0, 0);
    if (slot < 2 && slot < n) {
        if (first) {
            if (slot == 0) pm2 = *reinterpret_cast<const uint4*>(state + c);
            pm1 = *reinterpret_cast<const uint4*>(state + TF_H + c);
        } else {
            const uint16_t* r1 = bcx + size_t(row_base - 1) * TF_CIN + c;
            pm1 = gate8(*reinterpret_cast<const uint4*>(r1), *reinterpret_cast<const uint4*>(r1 + 2 * TF_H));
            if (slot == 0) {
                const uint16_t* r2 = bcx + size_t(row_base - 2) * TF_CIN + c;
                pm2 = gate8(*reinterpret_cast<const uint4*>(r2), *reinterpret_cast<const uint4*>(r2 + 2 * TF_H));
            }
        }
    }
    // a window that continues past its first tile: its last two entries (the new state)
    uint4 nl2 = make_uint4(0, 0, 0, 0), nl1 = make_uint4(0, 0, 0, 0);
    const bool writes_state = first && slot == 0;
    if (writes_state && st.rows > n) {
        const uint16_t* r2 = bcx + size_t(st.row_offset + st.rows - 2) * TF_CIN + c;
        const uint16_t* r1 = bcx + size_t(st.row_offset + st.rows - 1) * TF_CIN + c;
        nl2 = gate8(*reinterpret_cast<const uint4*>(r2), *reinterpret_cast<const uint4*>(r2 + 2 * TF_H));
        nl1 = gate8(*reinterpret_cast<const uint4*>(r1), *reinterpret_cast<const uint4*>(r1 + 2 * TF_H));
    }
    pdl_trigger();

    uint4 bx[RPT];
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        const int j = slot + k * kSlots;
        if (j < n) {
            bx[k] = gate8(B[k], X[k]);
            sbx[j][grp] = bx[k];
        }
    }
    __syncthreads();   // every entry of the tile is in; every read of the old state is done
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        const int j = slot + k * kSlots;
        if (j < n) {
            const uint4 e0 = j >= 2 ? sbx[j - 2][grp] : (j == 1 ? pm1 : pm2);
            const uint4 e1 = j >= 1 ? sbx[j - 1][grp] : pm1;
            float o[8];
            conv8(wv, e0, e1, bx[k], C[k], o);
            float4* yp = reinterpret_cast<float4*>(y + size_t(row_base + j) * TF_H + c);
            __stcs(yp, make_float4(o[0], o[1], o[2], o[3]));
            __stcs(yp + 1, make_float4(o[4], o[5], o[6], o[7]));
            if (hist) *reinterpret_cast<uint4*>(hist + size_t(tile.row0 + j + 2) * TF_H + c) = bx[k];
        }
    }
    if (writes_state) {
        if (hist) {   // history rows 0, 1: the old state
            *reinterpret_cast<uint4*>(hist + c) = pm2;
            *reinterpret_cast<uint4*>(hist + TF_H + c) = pm1;
        }
        // new state = the last two entries of [state0, state1, bx_0 .. bx_{r-1}]
        uint4 n0 = nl2, n1 = nl1;
        if (st.rows <= n) {   // the window ends in this tile
            n0 = n >= 2 ? sbx[n - 2][grp] : pm1;
            n1 = sbx[n - 1][grp];
        }
        *reinterpret_cast<uint4*>(state + c) = n0;
        *reinterpret_cast<uint4*>(state + TF_H + c) = n1;
    }
}

}  // namespace
}  // namespace tf

extern "C" int tf_conv_rows(const tf_segments* seg, int conv_layer, const void* bcx,
                            const void* w, float* y, tf_cuda_stream stream) {
    using namespace tf;
    if (!seg) return TF_EINVAL;
    const SegTable& t = seg->dev;
    if (conv_layer < 0 || conv_layer >= t.n_conv) return TF_EINVAL;
    if (t.R == 0) return TF_OK;
    if (!bcx || !w || !y || !aligned16(bcx) || !aligned16(w) || !aligned16(y)) return TF_EINVAL;
    const uint16_t* in = static_cast<const uint16_t*>(bcx);
    const uint16_t* wt = static_cast<const uint16_t*>(w);
    // tiles of two rows or more on average, and few of them: one row per
    // thread over 128 channels a CTA (twice the CTAs, half the serial work;
    // measured faster while the grid stays within twice the SM count); else
    // two rows per thread over 256 channels
    if (t.R >= 2 * t.n_tiles && t.n_tiles * (TF_H / Split<1>::kChanPerCta) <= 2 * sm_count())
        return launch_pdl(conv_rows_kernel<1>, dim3(t.n_tiles, TF_H / Split<1>::kChanPerCta), dim3(kThreads), 0,
                          stream, t, conv_layer, in, wt, y);
    return launch_pdl(conv_rows_kernel<2>, dim3(t.n_tiles, TF_H / Split<2>::kChanPerCta), dim3(kThreads), 0,
                      stream, t, conv_layer, in, wt, y);
}
