// score_noalloc.cu -- kvc_score for callers that cannot allocate device
// memory.
//
// Some hosts hand a plugin only its input and output buffers: there is no
// workspace argument to fill, and the plugin may not call cudaMalloc itself
// (the host's caching allocator has already reserved the device's memory,
// and a cudaMalloc would synchronise the whole device in the middle of the
// host's schedule).  kvc_score needs scratch for its per-row softmax
// statistics, so this entry point takes that scratch from a fixed array in
// the library's own device memory instead of a caller workspace.
//
// The array is a file-scope __device__ object of kStaticScratchBytes (8 MiB).
// It exists once per GPU that loads the library and stays resident until the
// process exits.  Host code cannot use the array's name as a device address
// (in host code it names a host-side stand-in), so the first call on each
// device looks the real address up with cudaGetSymbolAddress while that
// device is current, checks the result, and caches it; make that first call
// outside any stream capture.  Every call on a device shares the one array
// and leaves its contents behind: the device status word is cleared at the
// start of each call, everything else is fully rewritten before it is read.
// Two calls that overlap on the GPU (different streams, no ordering between
// them) race on the array and produce undefined scores -- order them on one
// stream or use kvc_score with separate workspaces.
//
// The kernels are the same ones kvc_score launches; only where their scratch
// lives differs.  Nothing here allocates: no cudaMalloc/cudaFree and no
// allocating library call.
#include "kvc_internal.cuh"

#include <mutex>

namespace kvc {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_score_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;

struct ScratchSlot {
    bool ready = false;
    unsigned char *ptr = nullptr;
};

// Device address of g_score_scratch on the current device (looked up once).
int scratch_address(unsigned char **out) {
    static std::mutex mu;
    static ScratchSlot slots[kMaxDevices];
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_error("kvc_score_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        set_error("kvc_score_noalloc: device index %d out of range", dev);
        return KVC_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (!slots[dev].ready) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_score_scratch);
        if (e != cudaSuccess || p == nullptr) {
            set_error("kvc_score_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
            return KVC_ERR_CUDA;
        }
        slots[dev].ptr = static_cast<unsigned char *>(p);
        slots[dev].ready = true;
    }
    *out = slots[dev].ptr;
    return KVC_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace kvc

using namespace kvc;

extern "C" int kvc_score_noalloc(const kvc_shape *shape, const void *q_obs, const void *k,
                                 float *scores, uint32_t *dev_status, cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_score_noalloc");
    // Same shape rules, kernel choice (KVC_SCORE_IMPL included) and work
    // split as kvc_score, so both entry points run the same kernels.
    if (!shape_ok(shape, "kvc_score_noalloc")) return KVC_ERR_INVALID_ARG;
    const kvc_shape &s = *shape;
    if (!q_obs || !k || !scores) {
        set_error("kvc_score_noalloc: NULL tensor");
        return KVC_ERR_INVALID_ARG;
    }
    if ((reinterpret_cast<uintptr_t>(q_obs) | reinterpret_cast<uintptr_t>(k)) & 15) {
        set_error("kvc_score_noalloc: q_obs and k must be 16-byte aligned");
        return KVC_ERR_INVALID_ARG;
    }
    // the kernels OR status bits into *dev_status with 32-bit atomics
    if (reinterpret_cast<uintptr_t>(dev_status) & 3) {
        set_error("kvc_score_noalloc: dev_status must be 4-byte aligned");
        return KVC_ERR_INVALID_ARG;
    }
    const int choice = score_impl_choice();
    if (choice < 0) {
        set_error("kvc_score_noalloc: KVC_SCORE_IMPL must be auto, simt or tc");
        return KVC_ERR_INVALID_ARG;
    }
    const bool can_tc = tc_eligible(s);
    if (choice == 2 && !can_tc) {
        set_error("kvc_score_noalloc: tensor-core path needs bf16, head_dim 64/128, G*W <= 512 "
                  "and an sm_100-family device");
        return KVC_ERR_UNSUPPORTED;
    }
    const bool tc = can_tc && choice != 1;
    const ScoreSplit sp = make_split(s, tc);

    const size_t partial_bytes = round256((size_t)sp.n_units * sp.max_slots * sp.rows_pad * sizeof(float2));
    const size_t bias_bytes = round256((size_t)sp.n_units * sp.rows_pad * sizeof(float));
    const size_t need = kWsHeader + partial_bytes + bias_bytes;
    if (need > kStaticScratchBytes) {
        set_error("kvc_score_noalloc: this shape needs %zu bytes of scratch, more than the %zu-byte "
                  "static buffer; use kvc_score with a workspace",
                  need, kStaticScratchBytes);
        return KVC_ERR_UNSUPPORTED;
    }

    unsigned char *scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc != KVC_OK) return rc;

    uint32_t *status = dev_status ? dev_status : reinterpret_cast<uint32_t *>(scratch);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) {
        set_error("kvc_score_noalloc: clearing the status word failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    ScoreArgs a;
    a.q = q_obs;
    a.k = k;
    a.scores = scores;
    a.partial = reinterpret_cast<float2 *>(scratch + kWsHeader);
    a.neg_bias = reinterpret_cast<float *>(scratch + kWsHeader + partial_bytes);
    a.status = status;
    return tc ? launch_score_tc(s, sp, a, stream) : launch_score_simt(s, sp, a, stream);
}
