// a5: greedy verify of every stream's window and the conv-state rewind.
//
// PR #1391 "lfm2: draft with LiquidAI's DSpark drafter (--drafter)": the
// target checks every draft, so a reply with drafts is the same as one without.
// PR #1377 "LFM2: shared-round decode", commit "a verify's greedy rows take the
// GPU's pick of their logits": a greedy row takes the GPU's pick, and the host
// samples a flagged row itself.
//
// Reading: draft j+1 is accepted while rows 0..j are accepted, row j is not
// flagged and pick[j] == ids[j+1]; the token after the prefix is pick[a]
// (or -1, host draw, when row a is flagged); a draft id outside [0, vocab)
// never matches and is reported. The conv state of every layer is rewound to
// history rows a+1, a+2 -- the state after row a.
//
// One CTA per (stream, conv layer); every warp finds the prefix length in one
// round trip (lane j tests draft j + 1, a ballot gives the first rejected
// one: windows hold at most 16 rows), CTAs of layer 0 write the per-stream
// results.
#include "tf_internal.cuh"

namespace tf {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
accept_kernel(SegTable t, const int32_t* __restrict__ ids, const int32_t* __restrict__ pick,
              const uint8_t* __restrict__ flag, int vocab, int32_t* accept_len,
              int32_t* next_token, int32_t* new_keys, uint8_t* sflag, int rewind) {
    const int s = blockIdx.x;
    const int layer = blockIdx.y;
    const SegStream st = t.streams[s];
    const int o = st.row_offset;
    pdl_wait();
    pdl_trigger();

    const int lane = threadIdx.x & 31;
    bool ok = false, bad = false;
    if (lane < st.rows - 1) {   // draft lane + 1 against the pick of row lane
        const int d = ids[o + lane + 1];
        bad = d < 0 || d >= vocab;
        ok = !bad && !flag[o + lane] && pick[o + lane] == d;
    }
    const unsigned ok_mask = __ballot_sync(0xFFFFFFFFu, ok);
    const unsigned bad_mask = __ballot_sync(0xFFFFFFFFu, bad);
    const int a = __ffs(~ok_mask) - 1;   // accepted drafts: the leading run (lane rows-1 is never ok)
    int sf = bad_mask ? 2 : 0;
    if (layer == 0 && threadIdx.x == 0) {
        int nxt = pick[o + a];
        if (flag[o + a]) {
            nxt = -1;
            sf |= 1;
        }
        accept_len[s] = a;
        next_token[s] = nxt;
        new_keys[s] = st.keys - st.rows + a + 1;
        sflag[s] = uint8_t(sf);
    }
    if (rewind && st.rows > 1 && layer < t.n_conv) {
        const size_t slot = size_t(layer) * t.S + s;
        const uint4* hist = static_cast<const uint4*>(t.conv_hist[slot]);
        uint4* state = static_cast<uint4*>(t.conv_state[slot]);
        constexpr int kRowVec = TF_H / 8;   // uint4 per row
        for (int k = threadIdx.x; k < 2 * kRowVec; k += kThreads)
            state[k] = hist[size_t(a + 1) * kRowVec + k];
    }
}

}  // namespace
}  // namespace tf

extern "C" int tf_accept(const tf_segments* seg, const int32_t* ids, const int32_t* pick,
                         const uint8_t* flag, int vocab, int32_t* accept_len, int32_t* next_token,
                         int32_t* new_keys, uint8_t* sflag, int rewind_conv, tf_cuda_stream stream) {
    using namespace tf;
    if (!seg || seg->prompt) return TF_EINVAL;
    const SegTable& t = seg->dev;
    if (t.S == 0) return TF_OK;
    if (!ids || !pick || !flag || !accept_len || !next_token || !new_keys || !sflag || vocab < 1)
        return TF_EINVAL;
    bool need_hist = false;
    for (const SegStream& st : seg->streams) need_hist |= st.rows > 1;
    if (rewind_conv && need_hist && t.n_conv > 0 && !t.has_hist) return TF_EINVAL;
    const int ly = (rewind_conv && t.n_conv > 0) ? t.n_conv : 1;
    dim3 grid(t.S, ly);
    return launch_pdl(accept_kernel, grid, dim3(kThreads), 0, stream, t, ids, pick, flag, vocab, accept_len,
                      next_token, new_keys, sflag, rewind_conv ? 1 : 0);
}
