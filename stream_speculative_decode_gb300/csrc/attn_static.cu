// tf_attn_static: one attention layer (partials, then merge) whose partial
// scratch is a fixed array compiled into the library, so the call allocates
// nothing.
//
// Who needs it: callers that cannot call cudaMalloc (or any allocating
// routine) at the point where they run attention -- code running under a
// custom allocator or a memory budget that forbids new device allocations,
// inside a memory pool they do not own, or a runtime that hands this library
// only the tensors it reads and writes. They pass the queries and the output;
// the scratch the split-K partials need lives in `g_partials` below.
//
// The array is a file-scope __device__ variable: every GPU on which this
// library's module is loaded holds TF_STATIC_SCRATCH_BYTES of it until the
// process exits. Its name is a host-side stand-in in host code, not a device
// address, so host code asks the runtime for the device address once per
// device (cudaGetSymbolAddress, with that device current) and passes that to
// the kernels.
#include <mutex>

#include "tf_internal.cuh"

namespace tf {
namespace {

static __device__ __align__(256) unsigned char g_partials[TF_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_partials_addr[kMaxDevices] = {nullptr};

// Device address of g_partials on the current device (set up on first use).
int partials_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return TF_ERANGE;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_partials_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_partials);
        if (e != cudaSuccess) return cuda_fail(e);
        g_partials_addr[dev] = p;
    }
    *out = g_partials_addr[dev];
    return TF_OK;
}

}  // namespace
}  // namespace tf

extern "C" int tf_attn_static(const tf_segments* seg, int attn_layer, const void* q, float* out,
                              tf_cuda_stream stream) {
    using namespace tf;
    if (!seg) return TF_EINVAL;
    const SegTable& t = seg->dev;
    if (attn_layer < 0 || attn_layer >= t.n_attn) return TF_EINVAL;
    if (seg->plan.partials_bytes > int64_t(TF_STATIC_SCRATCH_BYTES)) return TF_ERANGE;
    if (t.R == 0) return TF_OK;
    if (!q || !out || !aligned16(q) || !aligned16(out)) return TF_EINVAL;
    void* base = nullptr;
    int rc = partials_address(&base);
    if (rc != TF_OK) return rc;
    // Every record the merge reads is written by the partials launch first, so
    // nothing in the array has to start at zero.
    float* po = static_cast<float*>(base);
    float2* pml = reinterpret_cast<float2*>(po + t.n_partials * TF_D);
    rc = launch_attn_partials(t, attn_layer, static_cast<const uint16_t*>(q), po, pml, stream);
    if (rc != TF_OK) return rc;
    return launch_attn_merge(t, po, pml, out, stream);
}
