// Segment table: host validation, sizing and the device copy.
//
// PR #1377 "LFM2: shared-round decode", commit "a shared round runs each
// layer's conv and attention once over all its streams": the kernels run once
// a layer over every row, driven by a table that lists each stream's cache
// addresses, row offset and key count; streams longer than 8 rows are cut into
// tiles of 8; each stream keeps its own attention partials. The same commit's
// residency concern (a table reaching buffers nobody declared) becomes here a
// host check that the table's buffers are valid, aligned and never overlap.
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include <cudaTypedefs.h>   // PFN_cuTensorMapEncodeTiled

#include "tf_internal.cuh"

namespace tf {

static thread_local int g_last_cuda_error = 0;
static std::atomic<unsigned long long> g_wait_ns{TF_WAIT_LIMIT_DEFAULT_NS};

unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return TF_ECUDA;
}

int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        cache[dev] = n;
    }
    return cache[dev];
}

int attn_prepare();   // attn.cu: kernel attributes

namespace {

// cuTensorMapEncodeTiled, looked up once through the runtime (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// TMA map of one stream's K or V cache, bf16 [8][cap][64], as a 3-D tensor
// (d, key, head) of extents (64, keys, 8): keys past `keys` read as zeros. A box
// is 64 keys of one head, 128-byte rows, 128-byte swizzle (the layout the
// tensor-core kernel's shared-memory descriptors describe).
bool encode_kv_map(CUtensorMap* out, const void* base, int keys, int cap) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {cuuint64_t(TF_D), cuuint64_t(keys), cuuint64_t(TF_NKV)};
    const cuuint64_t strides[2] = {cuuint64_t(TF_D) * 2, cuuint64_t(cap) * TF_D * 2};
    const cuuint32_t box[3] = {cuuint32_t(TF_D), 64u, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool encode_q_map(CUtensorMap* out, const void* q, int rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    // (d, query head, row) of extents (64, 32, rows); a box is 4 heads of 4 rows
    // (16 query rows of 128 bytes), 128-byte swizzle; rows past `rows` read as zeros
    const cuuint64_t dims[3] = {cuuint64_t(TF_D), cuuint64_t(TF_NQ), cuuint64_t(rows)};
    const cuuint64_t strides[2] = {cuuint64_t(TF_D) * 2, cuuint64_t(TF_NQ) * TF_D * 2};
    const cuuint32_t box[3] = {cuuint32_t(TF_D), 4u, 4u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_w2_map(CUtensorMap* out, const void* w2, int rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cuuint64_t(TF_MK), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(TF_MK) * 2};
    const cuuint32_t box[2] = {64u, 128u};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w2), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Attention kernel of a stream: tensor cores once its window holds 3 rows (12
// query rows per KV head); TF_ATTN_PATH=mma|tc forces one (tests compare both).
int attn_path_of(int rows) {
    if (rows > 16) return kAttnTc;   // prompt windows (17-32 rows): the tensor cores, whatever is forced
    const char* e = std::getenv("TF_ATTN_PATH");
    if (e && std::strcmp(e, "mma") == 0) return kAttnMma;
    if (e && std::strcmp(e, "tc") == 0) return kAttnTc;
    return rows >= kTcMinRows ? kAttnTc : kAttnMma;
}

namespace {

struct Interval {
    uintptr_t lo, hi;
};

// True when two of the intervals overlap (empty intervals are ignored).
bool any_overlap(std::vector<Interval>& v) {
    std::sort(v.begin(), v.end(), [](const Interval& a, const Interval& b) { return a.lo < b.lo; });
    for (size_t i = 1; i < v.size(); ++i)
        if (v[i].lo < v[i - 1].hi) return true;
    return false;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace
}  // namespace tf

namespace tf {

// The plan of a set of windows, each of at most `max_window_rows` rows
// (TF_MAX_ROWS for the verify tables, kPromptTileRows for a prompt call).
int plan_windows(const tf_stream* streams, int n_streams, tf_plan* out, int max_window_rows) {
    if (!out) return TF_EINVAL;
    std::memset(out, 0, sizeof(*out));
    if (n_streams < 0) return TF_EINVAL;
    if (n_streams > TF_MAX_STREAMS) return TF_ERANGE;
    if (n_streams > 0 && !streams) return TF_EINVAL;
    int64_t R = 0, parts = 0, items = 0, tiles = 0;
    int max_rows = 0;
    bool any_mma = false, any_tc = false, any_merge = false;
    for (int s = 0; s < n_streams; ++s) {
        const tf_stream& st = streams[s];
        if (st.rows < 1 || st.keys < 1 || st.kv_capacity < 1) return TF_EINVAL;
        if (st.rows > max_window_rows || st.kv_capacity > TF_MAX_KEYS) return TF_ERANGE;
        if (st.row_offset != R) return TF_EINVAL;          // packed, in order
        if (st.keys < st.rows || st.keys > st.kv_capacity) return TF_EINVAL;
        int64_t chunk = tf_chunk_keys(st.rows);
        int64_t nch = (st.keys + chunk - 1) / chunk;
        R += st.rows;
        parts += int64_t(st.rows) * TF_NQ * nch;
        items += nch;
        tiles += (st.rows + tf::kConvTileRows - 1) / tf::kConvTileRows;
        max_rows = std::max(max_rows, int(st.rows));
        (tf::attn_path_of(st.rows) == tf::kAttnTc ? any_tc : any_mma) = true;
        if (nch > 1 && 4 * st.rows * nch > tf::kMergeLastCtaMaxRecords) any_merge = true;
    }
    if (R > (1 << 24)) return TF_ERANGE;
    out->n_streams = n_streams;
    out->n_rows = int32_t(R);
    out->max_rows = max_rows;
    out->n_conv_tiles = int32_t(tiles);
    out->n_attn_items = int32_t(items);
    out->attn_kernels = int32_t(any_mma) + int32_t(any_tc);
    out->attn_merge_launch = int32_t(any_merge);
    out->n_partials = parts;
    out->partials_bytes = parts * TF_D * 4 + parts * 8;
    return TF_OK;
}

}  // namespace tf

namespace {

// The rest of a build, shared by the verify and the prompt tables: sort the
// attention items, lay out and upload the blob, encode the TMA maps. `seg`
// (with its plan) is owned here from now on: freed on failure.
int finish_build(tf_segments* seg, std::vector<tf::SegStream>& ss, std::vector<int32_t>& row_stream,
                 std::vector<tf::ConvTile>& tiles, std::vector<tf::AttnItem>& items,
                 const void* const* conv_state, const void* const* conv_hist, const void* const* k_cache,
                 const void* const* v_cache, int n_conv, int n_attn, tf_cuda_stream stream, tf_segments** out) {
    using namespace tf;
    const int S = int(ss.size());
    const int R = int(row_stream.size());
    const tf_plan& plan = seg->plan;
    int rc = TF_OK;
    // mma.sync streams wider than kMmaGroupRows rows: one item per group of
    // rows and chunk, the groups of a chunk next to each other
    {
        std::vector<AttnItem> groups;
        groups.reserve(items.size());
        for (SegStream& d : ss) d.n_qg = 1;
        for (const AttnItem& it : items) {
            SegStream& d = ss[it.stream];
            const int ng = attn_path_of(d.rows) == kAttnMma ? (d.rows + kMmaGroupRows - 1) / kMmaGroupRows : 1;
            d.n_qg = ng;
            for (int gi = 0; gi < ng; ++gi) groups.push_back({it.stream, it.chunk, 4 * kMmaGroupRows * gi, 0});
        }
        items.swap(groups);
    }
    // mma.sync items first, then tensor-core items; within each, largest
    // chunks first so the long work starts early in the grid
    std::stable_sort(items.begin(), items.end(), [&](const AttnItem& a, const AttnItem& b) {
        const int pa = attn_path_of(ss[a.stream].rows), pb = attn_path_of(ss[b.stream].rows);
        if (pa != pb) return pa < pb;
        auto len = [&](const AttnItem& it) {
            const SegStream& d = ss[it.stream];
            int lo = it.chunk * d.chunk_keys;
            int len_keys = std::min(d.keys, lo + d.chunk_keys) - lo;
            return int64_t(len_keys) * ((d.rows + 3) / 4 + 1);
        };
        return len(a) > len(b);
    });
    int n_items_mma = 0, mma_rows = 1;
    for (const AttnItem& it : items)
        if (attn_path_of(ss[it.stream].rows) == kAttnMma) {
            ++n_items_mma;
            mma_rows = std::max(mma_rows, std::min(ss[it.stream].rows - it.q0 / 4, kMmaGroupRows));
        }

    size_t off = 0;
    const size_t o_streams = off;  off = align_up(off + sizeof(SegStream) * S, 256);
    const size_t o_rows = off;     off = align_up(off + sizeof(int32_t) * R, 256);
    const size_t o_tiles = off;    off = align_up(off + sizeof(ConvTile) * tiles.size(), 256);
    const size_t o_items = off;    off = align_up(off + sizeof(AttnItem) * items.size(), 256);
    const size_t n_cp = size_t(n_conv) * S, n_ap = size_t(n_attn) * S;
    const size_t o_cs = off;       off = align_up(off + sizeof(void*) * n_cp, 256);
    const size_t o_ch = off;       off = align_up(off + (conv_hist ? sizeof(void*) * n_cp : 0), 256);
    const size_t o_k = off;        off = align_up(off + sizeof(void*) * n_ap, 256);
    const size_t o_v = off;        off = align_up(off + sizeof(void*) * n_ap, 256);
    const size_t n_maps = size_t(n_items_mma) < items.size() ? n_ap : 0;
    const size_t o_km = off;       off = align_up(off + sizeof(CUtensorMap) * n_maps, 256);
    const size_t o_vm = off;       off = align_up(off + sizeof(CUtensorMap) * n_maps, 256);
    const size_t o_ctr = off;      off = align_up(off + sizeof(int32_t) * n_ap * TF_NKV, 256);
    const size_t n_groups = (size_t(S) + 127) / 128;   // Markov step: 128 streams per group
    const size_t o_mkk = off;      off = align_up(off + sizeof(unsigned long long) * S, 256);
    const size_t o_mkf = off;      off = align_up(off + sizeof(uint32_t) * S, 256);
    const size_t o_mkc = off;      off = align_up(off + sizeof(uint32_t) * n_groups, 256);
    const size_t o_tcw = off;      off = align_up(off + sizeof(int32_t) * 2 * size_t(n_attn), 256);
    const size_t o_mks = off;      off = align_up(off + kMkSyncBytes, 256);
    const size_t n_tc_units = (items.size() - size_t(n_items_mma)) * TF_NKV;
    const size_t o_redo = off;     off = align_up(off + sizeof(int32_t) * (1 + n_tc_units), 256);
    const size_t o_st = off;       off = align_up(off + sizeof(uint32_t), 256);
    const size_t total = off;
    seg->scratch_off = o_ctr;      // counters .. status word: zero in the image
    seg->scratch_bytes = total - o_ctr;

    seg->host.assign(total, 0);
    unsigned char* h = seg->host.data();
    if (S) std::memcpy(h + o_streams, ss.data(), sizeof(SegStream) * S);
    if (R) std::memcpy(h + o_rows, row_stream.data(), sizeof(int32_t) * R);
    if (!tiles.empty()) std::memcpy(h + o_tiles, tiles.data(), sizeof(ConvTile) * tiles.size());
    if (!items.empty()) std::memcpy(h + o_items, items.data(), sizeof(AttnItem) * items.size());
    if (n_cp) std::memcpy(h + o_cs, conv_state, sizeof(void*) * n_cp);
    if (n_cp && conv_hist) std::memcpy(h + o_ch, conv_hist, sizeof(void*) * n_cp);
    if (n_ap) {
        std::memcpy(h + o_k, k_cache, sizeof(void*) * n_ap);
        std::memcpy(h + o_v, v_cache, sizeof(void*) * n_ap);
    }
    for (size_t i = 0; i < n_maps; ++i) {
        const SegStream& st = ss[i % S];
        CUtensorMap km, vm;   // aligned locals, copied into the image
        if (!encode_kv_map(&km, k_cache[i], st.keys, st.cap) ||
            !encode_kv_map(&vm, v_cache[i], st.keys, st.cap)) {
            delete seg;
            return cuda_fail(cudaErrorInvalidValue);
        }
        std::memcpy(h + o_km + i * sizeof(CUtensorMap), &km, sizeof(CUtensorMap));
        std::memcpy(h + o_vm + i * sizeof(CUtensorMap), &vm, sizeof(CUtensorMap));
    }
    seg->streams = ss;

    SegTable& t = seg->dev;
    std::memset(&t, 0, sizeof(t));
    t.S = S;
    t.R = R;
    t.n_tiles = int32_t(tiles.size());
    t.n_items = int32_t(items.size());
    t.n_conv = n_conv;
    t.n_attn = n_attn;
    t.max_rows = plan.max_rows;
    t.has_hist = conv_hist ? 1 : 0;
    t.n_partials = plan.n_partials;
    t.n_items_mma = n_items_mma;
    t.mma_mt = (mma_rows + 3) / 4;
    t.n_merge_rows = 0;
    for (const SegStream& d : ss)
        if (d.merge_mode == kMergeKernel) t.n_merge_rows += d.rows;

    if (total > 0 && S > 0) {
        cudaError_t e = cudaMalloc(&seg->blob, total);
        if (e != cudaSuccess) {
            delete seg;
            cuda_fail(e);
            return e == cudaErrorMemoryAllocation ? TF_ENOMEM : TF_ECUDA;
        }
        e = cudaMemcpyAsync(seg->blob, h, total, cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) {
            cudaFree(seg->blob);
            delete seg;
            return cuda_fail(e);
        }
        unsigned char* b = static_cast<unsigned char*>(seg->blob);
        t.streams = reinterpret_cast<const SegStream*>(b + o_streams);
        t.row_stream = reinterpret_cast<const int32_t*>(b + o_rows);
        t.tiles = reinterpret_cast<const ConvTile*>(b + o_tiles);
        t.items = reinterpret_cast<const AttnItem*>(b + o_items);
        t.conv_state = reinterpret_cast<void* const*>(b + o_cs);
        t.conv_hist = conv_hist ? reinterpret_cast<void* const*>(b + o_ch) : nullptr;
        t.k_cache = reinterpret_cast<const void* const*>(b + o_k);
        t.v_cache = reinterpret_cast<const void* const*>(b + o_v);
        t.k_maps = n_maps ? reinterpret_cast<const CUtensorMap*>(b + o_km) : nullptr;
        t.v_maps = n_maps ? reinterpret_cast<const CUtensorMap*>(b + o_vm) : nullptr;
        t.counters = reinterpret_cast<int32_t*>(b + o_ctr);   // zero in the image
        t.mk_keys = reinterpret_cast<unsigned long long*>(b + o_mkk);   // zero in the image
        t.mk_flags = reinterpret_cast<uint32_t*>(b + o_mkf);
        t.mk_ctr = reinterpret_cast<uint32_t*>(b + o_mkc);
        t.tc_work = reinterpret_cast<int32_t*>(b + o_tcw);   // zero in the image
        t.mk_sync = reinterpret_cast<uint32_t*>(b + o_mks);
        t.tc_redo = reinterpret_cast<int32_t*>(b + o_redo);   // zero in the image
        t.status = reinterpret_cast<uint32_t*>(b + o_st);   // zero in the image
        rc = attn_prepare();
        if (rc == TF_OK) rc = attn_tc_prepare();
        if (rc == TF_OK && n_items_mma > 0 && size_t(n_items_mma) < items.size()) {
            // a round of both window kinds: the tensor-core launch runs on a side
            // stream with a grid proportional to its share of the keys (the K/V
            // bytes), the mma.sync launch takes the rest of the SMs
            int64_t keys_tc = 0, keys_all = 0;
            for (const SegStream& d : ss) {
                keys_all += d.keys;
                if (attn_path_of(d.rows) == kAttnTc) keys_tc += d.keys;
            }
            const int slots = 2 * sm_count();
            int g = int((int64_t(slots) * keys_tc + keys_all - 1) / (keys_all > 0 ? keys_all : 1));
            t.tc_grid_mixed = g < 1 ? 1 : (g > slots ? slots : g);
            if (cudaStreamCreateWithFlags(&t.side, cudaStreamNonBlocking) != cudaSuccess ||
                cudaEventCreateWithFlags(&t.ev_fork, cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&t.ev_join, cudaEventDisableTiming) != cudaSuccess) {
                // fall back to the two launches one after the other on the caller's stream
                if (t.ev_fork) cudaEventDestroy(t.ev_fork);
                if (t.side) cudaStreamDestroy(t.side);
                t.side = nullptr;
                t.ev_fork = t.ev_join = nullptr;
                cudaGetLastError();
            }
        }
        if (rc != TF_OK) {
            cudaFree(seg->blob);
            delete seg;
            return rc;
        }
    }
    *out = seg;
    return TF_OK;
}

}  // namespace

extern "C" {

int32_t tf_chunk_keys(int32_t rows) {
    if (rows >= tf::kTcMinRows && rows <= TF_MAX_ROWS) return 512 * rows;   // verify windows on the tensor-core kernel
    return 256 * (rows < 4 ? 4 : rows);
}

int tf_segments_plan(const tf_stream* streams, int n_streams, tf_plan* out) {
    return tf::plan_windows(streams, n_streams, out, TF_MAX_ROWS);
}

int tf_segments_build(const tf_stream* streams, int n_streams,
                      const void* const* conv_state, const void* const* conv_hist,
                      const void* const* k_cache, const void* const* v_cache,
                      int n_conv, int n_attn, tf_cuda_stream stream, tf_segments** out) {
    using namespace tf;
    if (!out) return TF_EINVAL;
    *out = nullptr;
    if (n_conv < 0 || n_attn < 0 || n_conv > 4096 || n_attn > 4096) return TF_EINVAL;
    tf_plan plan;
    int rc = tf_segments_plan(streams, n_streams, &plan);
    if (rc != TF_OK) return rc;
    const int S = n_streams;
    if (S > 0 && n_conv > 0 && !conv_state) return TF_EINVAL;
    if (S > 0 && n_attn > 0 && (!k_cache || !v_cache)) return TF_EINVAL;

    // ---- pointer checks: non-null, 16-byte aligned, no two buffers overlap
    std::vector<Interval> conv_iv, kv_iv;
    for (int l = 0; l < n_conv; ++l) {
        for (int s = 0; s < S; ++s) {
            const void* p = conv_state[size_t(l) * S + s];
            if (!p || !aligned16(p)) return TF_EINVAL;
            uintptr_t a = reinterpret_cast<uintptr_t>(p);
            conv_iv.push_back({a, a + size_t(2) * TF_H * 2});
            if (conv_hist) {
                const void* h = conv_hist[size_t(l) * S + s];
                if (!h) {
                    if (streams[s].rows > 1) return TF_EINVAL;
                    continue;
                }
                if (!aligned16(h)) return TF_EINVAL;
                uintptr_t b = reinterpret_cast<uintptr_t>(h);
                conv_iv.push_back({b, b + size_t(streams[s].rows + 2) * TF_H * 2});
            }
        }
    }
    for (int l = 0; l < n_attn; ++l) {
        for (int s = 0; s < S; ++s) {
            const void* k = k_cache[size_t(l) * S + s];
            const void* v = v_cache[size_t(l) * S + s];
            if (!k || !v || !aligned16(k) || !aligned16(v)) return TF_EINVAL;
            size_t bytes = size_t(TF_NKV) * streams[s].kv_capacity * TF_D * 2;
            uintptr_t a = reinterpret_cast<uintptr_t>(k), b = reinterpret_cast<uintptr_t>(v);
            kv_iv.push_back({a, a + bytes});
            kv_iv.push_back({b, b + bytes});
        }
    }
    if (any_overlap(conv_iv) || any_overlap(kv_iv)) return TF_EINVAL;

    tf_segments* seg = new (std::nothrow) tf_segments();
    if (!seg) return TF_ENOMEM;
    seg->plan = plan;
    const int R = plan.n_rows;

    // ---- host image: streams | row_stream | tiles | items | pointer arrays
    std::vector<SegStream> ss(S);
    std::vector<int32_t> row_stream(R);
    std::vector<ConvTile> tiles;
    std::vector<AttnItem> items;
    int64_t pbase = 0;
    for (int s = 0; s < S; ++s) {
        const tf_stream& st = streams[s];
        SegStream& d = ss[s];
        d.rows = st.rows;
        d.row_offset = st.row_offset;
        d.keys = st.keys;
        d.cap = st.kv_capacity;
        d.chunk_keys = tf_chunk_keys(st.rows);
        d.n_chunks = (st.keys + d.chunk_keys - 1) / d.chunk_keys;
        d.pbase = pbase;
        pbase += int64_t(st.rows) * TF_NQ * d.n_chunks;
        d.merge_mode = d.n_chunks == 1 ? kMergeDirect
                     : (4 * st.rows * d.n_chunks <= kMergeLastCtaMaxRecords ? kMergeLastCta : kMergeKernel);
        d.n_qg = 1;
        for (int i = 0; i < st.rows; ++i) row_stream[st.row_offset + i] = s;
        for (int r0 = 0; r0 < st.rows; r0 += kConvTileRows)
            tiles.push_back({s, r0, std::min(kConvTileRows, st.rows - r0), 0});
        for (int c = 0; c < d.n_chunks; ++c) items.push_back({s, c, 0, 0});
    }
    return finish_build(seg, ss, row_stream, tiles, items, conv_state, conv_hist, k_cache, v_cache, n_conv, n_attn,
                        stream, out);
}

int tf_prompt_build(int32_t rows, int32_t keys, int32_t kv_capacity, const void* const* conv_state,
                    const void* const* k_cache, const void* const* v_cache, int n_conv, int n_attn,
                    tf_cuda_stream stream, tf_segments** out) {
    using namespace tf;
    if (!out) return TF_EINVAL;
    *out = nullptr;
    if (n_conv < 0 || n_attn < 0 || n_conv > 4096 || n_attn > 4096) return TF_EINVAL;
    if (rows < 1 || keys < rows || kv_capacity < keys) return TF_EINVAL;
    if (rows > TF_MAX_PROMPT_ROWS || kv_capacity > TF_MAX_KEYS) return TF_ERANGE;
    if ((n_conv > 0 && !conv_state) || (n_attn > 0 && (!k_cache || !v_cache))) return TF_EINVAL;
    std::vector<Interval> conv_iv, kv_iv;
    for (int l = 0; l < n_conv; ++l) {
        const void* p = conv_state[l];
        if (!p || !aligned16(p)) return TF_EINVAL;
        const uintptr_t a = reinterpret_cast<uintptr_t>(p);
        conv_iv.push_back({a, a + size_t(2) * TF_H * 2});
    }
    const size_t kv_bytes = size_t(TF_NKV) * kv_capacity * TF_D * 2;
    for (int l = 0; l < n_attn; ++l) {
        const void* k = k_cache[l];
        const void* v = v_cache[l];
        if (!k || !v || !aligned16(k) || !aligned16(v)) return TF_EINVAL;
        const uintptr_t a = reinterpret_cast<uintptr_t>(k), b = reinterpret_cast<uintptr_t>(v);
        kv_iv.push_back({a, a + kv_bytes});
        kv_iv.push_back({b, b + kv_bytes});
    }
    if (any_overlap(conv_iv) || any_overlap(kv_iv)) return TF_EINVAL;

    // stream 0: the conv's view (every row, one state); streams 1..T: the
    // attention's windows of kPromptTileRows rows, each with its own causal
    // count over the same cache
    const int T = (rows + kPromptTileRows - 1) / kPromptTileRows;
    const int S = 1 + T;
    std::vector<tf_stream> tiles_as_streams;
    for (int t = 0; t < T; ++t) {
        const int r = std::min(kPromptTileRows, rows - t * kPromptTileRows);
        tiles_as_streams.push_back({r, t * kPromptTileRows, keys - rows + t * kPromptTileRows + r, kv_capacity});
    }
    tf_plan plan;
    int rc = plan_windows(tiles_as_streams.data(), T, &plan, kPromptTileRows);   // the attention work
    if (rc != TF_OK) return rc;
    plan.n_streams = 1;
    plan.n_conv_tiles = (rows + kConvTileRows - 1) / kConvTileRows;

    tf_segments* seg = new (std::nothrow) tf_segments();
    if (!seg) return TF_ENOMEM;
    seg->plan = plan;
    seg->prompt = true;
    std::vector<SegStream> ss(S);
    std::vector<int32_t> row_stream(rows);
    std::vector<ConvTile> tiles;
    std::vector<AttnItem> items;
    ss[0] = {rows, 0, keys, kv_capacity, 0, 0, 0, kMergeDirect, 1};
    for (int r0 = 0; r0 < rows; r0 += kConvTileRows) tiles.push_back({0, r0, std::min(kConvTileRows, rows - r0), 0});
    int64_t pbase = 0;
    for (int t = 0; t < T; ++t) {
        const tf_stream& st = tiles_as_streams[t];
        SegStream& d = ss[1 + t];
        d.rows = st.rows;
        d.row_offset = st.row_offset;
        d.keys = st.keys;
        d.cap = st.kv_capacity;
        d.chunk_keys = tf_chunk_keys(st.rows);
        d.n_chunks = (st.keys + d.chunk_keys - 1) / d.chunk_keys;
        d.pbase = pbase;
        pbase += int64_t(st.rows) * TF_NQ * d.n_chunks;
        d.merge_mode = d.n_chunks == 1 ? kMergeDirect
                     : (4 * st.rows * d.n_chunks <= kMergeLastCtaMaxRecords ? kMergeLastCta : kMergeKernel);
        d.n_qg = 1;
        for (int i = 0; i < st.rows; ++i) row_stream[st.row_offset + i] = 1 + t;
        for (int c = 0; c < d.n_chunks; ++c) items.push_back({1 + t, c, 0, 0});
    }
    // pointer arrays [layer][S]: every stream of a layer names the layer's
    // state and caches (the conv reaches them through stream 0 only)
    std::vector<const void*> cs(size_t(n_conv) * S), kc(size_t(n_attn) * S), vc(size_t(n_attn) * S);
    for (int l = 0; l < n_conv; ++l)
        for (int s = 0; s < S; ++s) cs[size_t(l) * S + s] = conv_state[l];
    for (int l = 0; l < n_attn; ++l)
        for (int s = 0; s < S; ++s) {
            kc[size_t(l) * S + s] = k_cache[l];
            vc[size_t(l) * S + s] = v_cache[l];
        }
    return finish_build(seg, ss, row_stream, tiles, items, n_conv ? cs.data() : nullptr, nullptr,
                        n_attn ? kc.data() : nullptr, n_attn ? vc.data() : nullptr, n_conv, n_attn, stream, out);
}

int tf_segments_free(tf_segments* seg) {
    if (!seg) return TF_OK;
    int rc = TF_OK;
    if (seg->dev.ev_join) cudaEventDestroy(seg->dev.ev_join);
    if (seg->dev.ev_fork) cudaEventDestroy(seg->dev.ev_fork);
    if (seg->dev.side) cudaStreamDestroy(seg->dev.side);
    if (seg->blob) {
        cudaError_t e = cudaFree(seg->blob);
        if (e != cudaSuccess) rc = tf::cuda_fail(e);
    }
    delete seg;
    return rc;
}

int tf_segments_query(const tf_segments* seg, tf_plan* out) {
    if (!seg || !out) return TF_EINVAL;
    *out = seg->plan;
    return TF_OK;
}

size_t tf_partials_bytes(const tf_segments* seg) {
    return seg ? size_t(seg->plan.partials_bytes) : 0;
}

const char* tf_strerror(int status) {
    switch (status) {
        case TF_OK: return "TF_OK: success";
        case TF_EINVAL: return "TF_EINVAL: invalid argument (null, shape, packing, alignment or aliasing)";
        case TF_ERANGE: return "TF_ERANGE: size out of the supported range";
        case TF_ENOMEM: return "TF_ENOMEM: device allocation of the segment table failed";
        case TF_ECUDA: return "TF_ECUDA: a CUDA call or kernel launch failed";
        case TF_ETIMEOUT: return "TF_ETIMEOUT: a kernel gave up a bounded device wait; the table's results since the "
                                 "last check are not valid";
        default: return "unknown tf status";
    }
}

int tf_last_cuda_error(void) { return tf::g_last_cuda_error; }

int tf_set_wait_limit_ns(uint64_t ns) {
    if (ns > TF_WAIT_LIMIT_MAX_NS) return TF_ERANGE;
    tf::g_wait_ns.store(ns);
    return TF_OK;
}

uint64_t tf_wait_limit_ns(void) { return tf::g_wait_ns.load(); }

int tf_segments_status(tf_segments* seg, tf_cuda_stream stream, uint32_t* bits) {
    if (bits) *bits = 0;
    if (!seg) return TF_EINVAL;
    if (!seg->blob) return TF_OK;   // an empty round launches nothing
    uint32_t h = 0;
    cudaError_t e = cudaMemcpyAsync(&h, seg->dev.status, sizeof(h), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return tf::cuda_fail(e);
    if (bits) *bits = h;
    if (h == 0) return TF_OK;
    // a CTA that gave up may have left the cross-CTA counters and merge
    // scratch mid-count: back to the image's zeros, status word included
    e = cudaMemsetAsync(static_cast<unsigned char*>(seg->blob) + seg->scratch_off, 0, seg->scratch_bytes, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return tf::cuda_fail(e);
    return TF_ETIMEOUT;
}

}  // extern "C"
