// The next verify's ids, written on the GPU from each stream's pending token
// and the drafter's picks (no host round trip between the drafter and the
// verify).
//
// PR #1391 "lfm2: draft with LiquidAI's DSpark drafter (--drafter)", the held
// path: a kernel fills each verify window's ids from the drafter's picks;
// after review, a nonfinite pick or an id past the vocabulary is no longer
// turned into token 0 but raises a flag that the verify checks.
//
// Layout (reading): window row 0 of stream s is its pending token prev[s];
// window row j >= 1 is the draft at packed draft row o_s - s + j - 1 (each
// stream contributes rows_s - 1 drafts, stream after stream). A bad token is
// written as -1, which the verify never accepts, and sets the stream's flag:
// bit 0 for the pending token, bit 1 for a draft.
//
// One warp per stream, one lane per window row (rows <= 16); the flag is a
// warp ballot. Pure copy: 4 bytes in, 4 bytes out per row.
#include "tf_internal.cuh"

namespace tf {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
draft_ids_kernel(SegTable t, const int32_t* __restrict__ prev, const int32_t* __restrict__ drafts,
                 const uint8_t* __restrict__ draft_flag, int vocab, int32_t* __restrict__ ids,
                 uint8_t* __restrict__ dflag) {
    const int s = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    pdl_wait();   // the pending tokens and picks may come from the kernels just before
    if (s >= t.S) return;
    const SegStream st = t.streams[s];
    bool bad_pending = false, bad_draft = false;
    if (lane < st.rows) {
        int tok;
        bool bad;
        if (lane == 0) {
            tok = prev[s];
            bad = tok < 0 || tok >= vocab;
            bad_pending = bad;
        } else {
            const int k = st.row_offset - s + lane - 1;
            tok = drafts[k];
            bad = tok < 0 || tok >= vocab || (draft_flag && draft_flag[k]);
            bad_draft = bad;
        }
        ids[st.row_offset + lane] = bad ? -1 : tok;
    }
    pdl_trigger();
    const unsigned bp = __ballot_sync(0xFFFFFFFFu, bad_pending);
    const unsigned bd = __ballot_sync(0xFFFFFFFFu, bad_draft);
    if (lane == 0) dflag[s] = uint8_t((bp ? 1 : 0) | (bd ? 2 : 0));
}

}  // namespace
}  // namespace tf

extern "C" int tf_draft_ids(const tf_segments* seg, const int32_t* prev, const int32_t* drafts,
                            const uint8_t* draft_flag, int vocab, int32_t* ids, uint8_t* dflag,
                            tf_cuda_stream stream) {
    using namespace tf;
    if (!seg || seg->prompt) return TF_EINVAL;
    const SegTable& t = seg->dev;
    if (t.S == 0) return TF_OK;
    if (!prev || !ids || !dflag || vocab < 1) return TF_EINVAL;
    if (!drafts && t.R > t.S) return TF_EINVAL;   // some window holds drafts
    const dim3 grid((t.S + kWarps - 1) / kWarps);
    return launch_pdl(draft_ids_kernel, grid, dim3(kWarps * 32), 0, stream, t, prev, drafts, draft_flag, vocab,
                      ids, dflag);
}
