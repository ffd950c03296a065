// a1: LFM2 gated short conv over every row of every stream, one launch a layer.
//
// PR #1377 "LFM2: shared-round decode", commit "a shared round runs each
// layer's conv and attention once over all its streams": one launch a layer
// over every row from the segment table, each row's arithmetic that of the
// per-stream conv; streams longer than 8 rows are folded into 8-row tiles.
//
// Work split: a CTA of 64 threads owns one 8-row tile of one stream and 512
// channels; a thread owns 8 consecutive channels (16-byte loads of B, C, x and
// of the 3 taps) and walks the tile's rows in order. The two rows before a
// tile come from the conv state (first tile) or are recomputed from the
// input rows (later tiles), so tiles are independent. Only the first tile of a
// stream reads the state and only it writes the new state, so the in-place
// update needs no ordering between CTAs.
//
// HBM bound: per row 6144*2 B read + 2048*4 B written (+ state/history).
#include "tf_internal.cuh"

namespace tf {
namespace {

constexpr int kThreads = 64;
constexpr int kChan = 8;                       // channels per thread
constexpr int kChanPerCta = kThreads * kChan;  // 512

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

__global__ void __launch_bounds__(kThreads)
conv_rows_kernel(SegTable t, int layer, const uint16_t* __restrict__ bcx,
                 const uint16_t* __restrict__ w, float* __restrict__ y) {
    const ConvTile tile = t.tiles[blockIdx.x];
    const SegStream st = t.streams[tile.stream];
    const int c = blockIdx.y * kChanPerCta + threadIdx.x * kChan;
    const size_t slot = size_t(layer) * t.S + tile.stream;
    uint16_t* state = static_cast<uint16_t*>(t.conv_state[slot]);
    uint16_t* hist = t.has_hist ? static_cast<uint16_t*>(t.conv_hist[slot]) : nullptr;
    const int n = tile.nrows;
    const int row_base = st.row_offset + tile.row0;
    pdl_wait();   // the table above; the data below may come from the previous kernel

    // taps of channels c..c+7: 24 bf16, element (channel j, tap k) at 3*j+k
    float wt[24];
    {
        const uint4* wp = reinterpret_cast<const uint4*>(w + size_t(c) * 3);
        float a[8], b[8], d[8];
        unpack8(__ldg(wp + 0), a);
        unpack8(__ldg(wp + 1), b);
        unpack8(__ldg(wp + 2), d);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            wt[k] = a[k];
            wt[8 + k] = b[k];
            wt[16 + k] = d[k];
        }
    }

    // the window rows of this tile (loads issued before any arithmetic)
    uint4 B[kConvTileRows], C[kConvTileRows], X[kConvTileRows];
#pragma unroll
    for (int j = 0; j < kConvTileRows; ++j) {
        if (j < n) {
            const uint16_t* row = bcx + size_t(row_base + j) * TF_CIN + c;
            B[j] = __ldcs(reinterpret_cast<const uint4*>(row));
            C[j] = __ldcs(reinterpret_cast<const uint4*>(row + TF_H));
            X[j] = __ldcs(reinterpret_cast<const uint4*>(row + 2 * TF_H));
        }
    }

    // the two sequence entries before the tile
    uint4 s0, s1;
    if (tile.row0 == 0) {
        s0 = *reinterpret_cast<const uint4*>(state + c);
        s1 = *reinterpret_cast<const uint4*>(state + TF_H + c);
    } else {
        const uint16_t* r2 = bcx + size_t(row_base - 2) * TF_CIN + c;
        const uint16_t* r1 = bcx + size_t(row_base - 1) * TF_CIN + c;
        s0 = gate8(*reinterpret_cast<const uint4*>(r2), *reinterpret_cast<const uint4*>(r2 + 2 * TF_H));
        s1 = gate8(*reinterpret_cast<const uint4*>(r1), *reinterpret_cast<const uint4*>(r1 + 2 * TF_H));
    }
    const uint4 old0 = s0, old1 = s1;
    pdl_trigger();

    float f0[8], f1[8];
    unpack8(s0, f0);
    unpack8(s1, f1);
#pragma unroll
    for (int j = 0; j < kConvTileRows; ++j) {
        if (j < n) {
            const uint4 bx = gate8(B[j], X[j]);
            float f2[8], fc[8];
            unpack8(bx, f2);
            unpack8(C[j], fc);
            float o[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float conv = wt[3 * k] * f0[k];
                conv = fmaf(wt[3 * k + 1], f1[k], conv);
                conv = fmaf(wt[3 * k + 2], f2[k], conv);
                o[k] = fc[k] * conv;
            }
            float4* yp = reinterpret_cast<float4*>(y + size_t(row_base + j) * TF_H + c);
            __stcs(yp, make_float4(o[0], o[1], o[2], o[3]));
            __stcs(yp + 1, make_float4(o[4], o[5], o[6], o[7]));
            if (hist)
                *reinterpret_cast<uint4*>(hist + size_t(tile.row0 + j + 2) * TF_H + c) = bx;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                f0[k] = f1[k];
                f1[k] = f2[k];
            }
            s0 = s1;
            s1 = bx;
        }
    }

    if (tile.row0 == 0) {
        if (hist) {
            *reinterpret_cast<uint4*>(hist + c) = old0;
            *reinterpret_cast<uint4*>(hist + TF_H + c) = old1;
        }
        // new state = the last two entries of [state0, state1, bx_0 .. bx_{r-1}]
        uint4 n0 = s0, n1 = s1;
        if (st.rows > n) {   // the window continues in later tiles
            const uint16_t* r2 = bcx + size_t(st.row_offset + st.rows - 2) * TF_CIN + c;
            const uint16_t* r1 = bcx + size_t(st.row_offset + st.rows - 1) * TF_CIN + c;
            n0 = gate8(*reinterpret_cast<const uint4*>(r2), *reinterpret_cast<const uint4*>(r2 + 2 * TF_H));
            n1 = gate8(*reinterpret_cast<const uint4*>(r1), *reinterpret_cast<const uint4*>(r1 + 2 * TF_H));
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
    dim3 grid(t.n_tiles, TF_H / kChanPerCta);
    return launch_pdl(conv_rows_kernel, grid, dim3(kThreads), 0, stream, t, conv_layer,
                      static_cast<const uint16_t*>(bcx), static_cast<const uint16_t*>(w), y);
}
