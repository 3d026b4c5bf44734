// api.cu -- the extern "C" entry points of libkvc: argument validation,
// workspace layout and dispatch to the kernels.  Nothing here allocates
// device memory; every launch goes to the caller's stream.
#include "kvc_internal.cuh"

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

namespace kvc {

namespace {
thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct DeviceInfo {
    int sms = 0;
    int major = 0;
};

DeviceInfo device_info() {
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DeviceInfo{};
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev].sms == 0) {
        cudaDeviceGetAttribute(&cache[dev].sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&cache[dev].major, cudaDevAttrComputeCapabilityMajor, dev);
    }
    return cache[dev];
}

struct WsLayout {
    size_t partial_off, partial_bytes;
    size_t bias_off, bias_bytes;
    size_t vpart_off, vpart_bytes;   // THINKV per-part channel sums
    size_t vscore_off, vscore_bytes; // THINKV channel scores when the caller passes none
    size_t total;
};

WsLayout ws_layout(const kvc_shape &s) {
    const ScoreSplit a = make_split(s, true), b = make_split(s, false);
    const int slots = a.max_slots > b.max_slots ? a.max_slots : b.max_slots;
    WsLayout w;
    w.partial_off = kWsHeader;
    w.partial_bytes = align256((size_t)a.n_units * slots * a.rows_pad * sizeof(float2));
    w.bias_off = w.partial_off + w.partial_bytes;
    w.bias_bytes = align256((size_t)a.n_units * a.rows_pad * sizeof(float));
    w.vpart_off = w.bias_off + w.bias_bytes;
    w.vpart_bytes = align256((size_t)value_partial_floats(s) * sizeof(float));
    w.vscore_off = w.vpart_off + w.vpart_bytes;
    w.vscore_bytes = align256((size_t)a.n_units * s.head_dim * sizeof(float));
    w.total = w.vscore_off + w.vscore_bytes;
    return w;
}

bool ws_ok(void *ws, size_t ws_bytes, size_t need, const char *fn) {
    if (!ws) return fail(KVC_ERR_WORKSPACE, "%s: workspace is NULL", fn), false;
    if (ws_bytes < need)
        return fail(KVC_ERR_WORKSPACE, "%s: workspace has %zu bytes, needs %zu", fn, ws_bytes, need),
               false;
    if (reinterpret_cast<uintptr_t>(ws) % 256)
        return fail(KVC_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", fn), false;
    return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

uint32_t *status_word(void *ws) { return static_cast<uint32_t *>(ws); }
// Completion counter of the MBA launch (zero between launches).
uint32_t *mba_done_word(void *ws) { return static_cast<uint32_t *>(ws) + 1; }


// Event sets of kvc_compress_host, one per (device, staging buffer); created
// on first use and kept (at most kMaxEventSets idle sets; the oldest idle set
// is destroyed when a new buffer needs one and the cache is full).
struct EventSet {
    int dev = -1;
    const void *key = nullptr;
    bool in_use = false;
    unsigned long long last_use = 0;
    std::vector<cudaEvent_t> layer;
    cudaEvent_t last_done = nullptr;
};
constexpr size_t kMaxEventSets = 64;
std::mutex g_ev_mu;
std::vector<EventSet *> g_ev_sets;
unsigned long long g_ev_clock = 0;

// An evicted set is destroyed only after its last call has finished reading
// its staging buffers, so a later call on the same buffers (which gets a
// fresh set) cannot overwrite them early.
void destroy_set(EventSet *e) {
    if (e->last_done) cudaEventSynchronize(e->last_done);
    for (cudaEvent_t x : e->layer) cudaEventDestroy(x);
    if (e->last_done) cudaEventDestroy(e->last_done);
    delete e;
}

int checkout_events(const void *key, int n_layer_events, EventSet **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return fail(KVC_ERR_CUDA, "kvc_compress_host: cudaGetDevice failed");
    std::lock_guard<std::mutex> lk(g_ev_mu);
    EventSet *e = nullptr;
    for (EventSet *c : g_ev_sets)
        if (c->dev == dev && c->key == key) e = c;
    if (e && e->in_use)
        return fail(KVC_ERR_INVALID_ARG,
                    "kvc_compress_host: another call is using these staging buffers right now");
    if (!e) {
        if (g_ev_sets.size() >= kMaxEventSets) {
            size_t victim = g_ev_sets.size();
            for (size_t i = 0; i < g_ev_sets.size(); ++i)
                if (!g_ev_sets[i]->in_use &&
                    (victim == g_ev_sets.size() || g_ev_sets[i]->last_use < g_ev_sets[victim]->last_use))
                    victim = i;
            if (victim < g_ev_sets.size()) {
                destroy_set(g_ev_sets[victim]);
                g_ev_sets.erase(g_ev_sets.begin() + (long)victim);
            }
        }
        e = new EventSet;
        e->dev = dev;
        e->key = key;
        if (cudaEventCreateWithFlags(&e->last_done, cudaEventDisableTiming) != cudaSuccess) {
            delete e;
            return fail(KVC_ERR_CUDA, "kvc_compress_host: cudaEventCreate failed");
        }
        g_ev_sets.push_back(e);
    }
    while ((int)e->layer.size() < n_layer_events) {
        cudaEvent_t x;
        if (cudaEventCreateWithFlags(&x, cudaEventDisableTiming) != cudaSuccess)
            return fail(KVC_ERR_CUDA, "kvc_compress_host: cudaEventCreate failed");
        e->layer.push_back(x);
    }
    e->in_use = true;
    e->last_use = ++g_ev_clock;
    *out = e;
    return KVC_OK;
}

void checkin_events(EventSet *e) {
    std::lock_guard<std::mutex> lk(g_ev_mu);
    e->in_use = false;
}

// The window rows' softmax statistics a plain score pass leaves in a
// workspace (the merge's -(m_r + log2 l_r)), recorded per workspace with what
// they were computed from, so that kvc_channel_prune_value_ex can reuse them
// on request.  Host-side and per process; a record is replaced by the next
// plain score pass over the workspace and dropped by anything else that
// rewrites the statistics (a Keyformer score, a workspace reset).
struct StatsRecord {
    const void *ws;
    kvc_shape s;
    const void *q, *k;
    bool tc;
    int device;
};
std::mutex g_stats_mu;
std::vector<StatsRecord> g_stats;

bool same_shape(const kvc_shape &a, const kvc_shape &b) {
    return a.n_layers == b.n_layers && a.n_q_heads == b.n_q_heads && a.n_kv_heads == b.n_kv_heads &&
           a.head_dim == b.head_dim && a.seq_len == b.seq_len && a.window == b.window &&
           a.dtype == b.dtype;
}

int current_device() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess) {
        cudaGetLastError();
        d = -1;
    }
    return d;
}

void stats_forget(const void *ws) {
    std::lock_guard<std::mutex> lk(g_stats_mu);
    for (size_t i = 0; i < g_stats.size(); ++i)
        if (g_stats[i].ws == ws) {
            g_stats[i] = g_stats.back();
            g_stats.pop_back();
            return;
        }
}

void stats_record(const void *ws, const kvc_shape &s, const void *q, const void *k, bool tc) {
    const StatsRecord r{ws, s, q, k, tc, current_device()};
    std::lock_guard<std::mutex> lk(g_stats_mu);
    for (auto &e : g_stats)
        if (e.ws == ws) {
            e = r;
            return;
        }
    g_stats.push_back(r);
}

bool stats_match(const void *ws, const kvc_shape &s, const void *q, const void *k, bool tc) {
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_stats_mu);
    for (const auto &e : g_stats)
        if (e.ws == ws)
            return same_shape(e.s, s) && e.q == q && e.k == k && e.tc == tc && e.device == dev;
    return false;
}

}  // namespace

// Shape validation and score-kernel choice, shared by every entry point that
// scores (kvc_score, kvc_score_keyformer, kvc_score_noalloc).
bool shape_ok(const kvc_shape *s, const char *fn) {
    if (!s) return fail(KVC_ERR_INVALID_ARG, "%s: shape is NULL", fn), false;
    if (s->n_layers < 1 || s->n_q_heads < 1 || s->n_kv_heads < 1)
        return fail(KVC_ERR_INVALID_ARG, "%s: layers and heads must be >= 1", fn), false;
    if (s->n_q_heads % s->n_kv_heads)
        return fail(KVC_ERR_INVALID_ARG, "%s: n_q_heads %% n_kv_heads != 0", fn), false;
    if (s->head_dim < 1 || s->head_dim > 256)
        return fail(KVC_ERR_INVALID_ARG, "%s: head_dim must be in 1..256", fn), false;
    if (s->window < 1 || s->seq_len <= s->window)
        return fail(KVC_ERR_INVALID_ARG, "%s: need 1 <= window < seq_len", fn), false;
    if (s->dtype != KVC_F32 && s->dtype != KVC_BF16)
        return fail(KVC_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, s->dtype), false;
    if ((int64_t)s->n_layers * s->n_kv_heads > (1 << 30))
        return fail(KVC_ERR_INVALID_ARG, "%s: too many heads", fn), false;
    return true;
}

bool tc_eligible(const kvc_shape &s) {
    const int G = s.n_q_heads / s.n_kv_heads;
    return s.dtype == KVC_BF16 && (s.head_dim == 64 || s.head_dim == 128) &&
           (int64_t)G * s.window <= kMaxRowsTC && device_info().major >= 10;
}

int score_impl_choice() {
    const char *e = getenv("KVC_SCORE_IMPL");
    if (!e || !*e || !strcmp(e, "auto")) return 0;
    if (!strcmp(e, "simt")) return 1;
    if (!strcmp(e, "tc")) return 2;
    return -1;
}

ScoreSplit make_split(const kvc_shape &s, bool tc) {
    const int sms = device_info().sms;
    return make_score_split(s, tc, sms, tc ? score_tc_pairs(sms) : 0);
}

void set_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
}

}  // namespace kvc

using namespace kvc;

extern "C" {

size_t kvc_workspace_size(const kvc_shape *shape, int32_t k_max) {
    (void)k_max;
    if (!shape_ok(shape, "kvc_workspace_size")) return 0;
    return ws_layout(*shape).total;
}

int kvc_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_workspace_init");
    g_err[0] = 0;
    if (!ws || ws_bytes < kWsHeader) return fail(KVC_ERR_WORKSPACE, "kvc_workspace_init: bad workspace");
    stats_forget(ws);
    cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, stream);
    if (e != cudaSuccess) return fail(KVC_ERR_CUDA, "kvc_workspace_init: %s", cudaGetErrorString(e));
    return KVC_OK;
}

int kvc_workspace_status(const void *ws, size_t ws_bytes, uint32_t *status, cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_workspace_status");
    g_err[0] = 0;
    if (!ws || ws_bytes < kWsHeader || !status)
        return fail(KVC_ERR_INVALID_ARG, "kvc_workspace_status: bad arguments");
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(KVC_ERR_CUDA, "kvc_workspace_status: %s", cudaGetErrorString(e));
    *status = v;
    return KVC_OK;
}

int kvc_score(const kvc_shape *shape, const void *q_obs, const void *k, float *scores, void *ws,
              size_t ws_bytes, cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_score");
    g_err[0] = 0;
    if (!shape_ok(shape, "kvc_score")) return KVC_ERR_INVALID_ARG;
    if (!q_obs || !k || !scores) return fail(KVC_ERR_INVALID_ARG, "kvc_score: NULL tensor");
    if (!aligned16(q_obs) || !aligned16(k))
        return fail(KVC_ERR_INVALID_ARG, "kvc_score: q_obs and k must be 16-byte aligned");
    const kvc_shape &s = *shape;
    const WsLayout w = ws_layout(s);
    if (!ws_ok(ws, ws_bytes, w.total, "kvc_score")) return KVC_ERR_WORKSPACE;
    const int choice = score_impl_choice();
    if (choice < 0) return fail(KVC_ERR_INVALID_ARG, "kvc_score: KVC_SCORE_IMPL must be auto, simt or tc");
    const bool can_tc = tc_eligible(s);
    if (choice == 2 && !can_tc)
        return fail(KVC_ERR_UNSUPPORTED, "kvc_score: tensor-core path needs bf16, head_dim 64/128, "
                                         "G*W <= 512 and an sm_100-family device");
    const bool tc = can_tc && choice != 1;
    const ScoreSplit sp = make_split(s, tc);
    ScoreArgs a;
    a.q = q_obs;
    a.k = k;
    a.scores = scores;
    a.partial = reinterpret_cast<float2 *>(static_cast<char *>(ws) + w.partial_off);
    a.neg_bias = reinterpret_cast<float *>(static_cast<char *>(ws) + w.bias_off);
    a.status = status_word(ws);
    const int rc = tc ? launch_score_tc(s, sp, a, stream) : launch_score_simt(s, sp, a, stream);
    if (rc == KVC_OK)
        stats_record(ws, s, q_obs, k, tc);
    else
        stats_forget(ws);
    return rc;
}

// Host-resident prompt, whole default path (see kvc.h).
int kvc_compress_host(const kvc_shape *shape, const void *q_host, const void *k_host,
                      const void *v_host, void *q_dev, void *k_dev, uint32_t mass_num,
                      uint32_t mass_den, int64_t total_budget, int32_t layer_floor, int32_t k_max,
                      float *scores, int32_t *mba, int32_t *budget, int32_t *idx, void *k_out,
                      void *v_out, int64_t out_rows, void *ws, size_t ws_bytes, cudaStream_t stream,
                      cudaStream_t copy_stream) {
    NvtxRange nvtx_range("kvc_compress_host");
    g_err[0] = 0;
    if (!shape_ok(shape, "kvc_compress_host")) return KVC_ERR_INVALID_ARG;
    const kvc_shape &s = *shape;
    if (!q_host || !k_host || !v_host || !q_dev || !k_dev || !scores || !mba || !budget || !idx ||
        !k_out || !v_out)
        return fail(KVC_ERR_INVALID_ARG, "kvc_compress_host: NULL pointer");
    if (stream == copy_stream)
        return fail(KVC_ERR_INVALID_ARG, "kvc_compress_host: copies need a stream of their own");
    if (!aligned16(q_dev) || !aligned16(k_dev) || !aligned16(k_out) || !aligned16(v_out))
        return fail(KVC_ERR_INVALID_ARG, "kvc_compress_host: device buffers must be 16-byte aligned");
    if (k_max < 1 || out_rows < 0) return fail(KVC_ERR_INVALID_ARG, "kvc_compress_host: bad k_max/out_rows");
    const WsLayout w = ws_layout(s);
    if (!ws_ok(ws, ws_bytes, w.total, "kvc_compress_host")) return KVC_ERR_WORKSPACE;
    // V is never copied: the compaction reads the kept rows through the
    // device's mapping of the (pinned) host buffer.  The mapping is looked up
    // in the calling thread's current context, which a thread that has not
    // made a runtime call yet does not have: bind the current device's
    // primary context first.
    {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) {
            cudaGetLastError();
            return fail(KVC_ERR_CUDA, "kvc_compress_host: no usable CUDA device");
        }
    }
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, v_host) != cudaSuccess || pa.type != cudaMemoryTypeHost ||
        pa.devicePointer == nullptr) {
        cudaGetLastError();
        return fail(KVC_ERR_INVALID_ARG,
                    "kvc_compress_host: v_host must be pinned host memory mapped for the device");
    }
    const void *v_dev = pa.devicePointer;
    if (!aligned16(v_dev)) return fail(KVC_ERR_INVALID_ARG, "kvc_compress_host: v_host must be 16-byte aligned");
    // One set of events per staging buffer (per device): an event per layer
    // of K plus one for Q, and `last_done`, recorded after the call's last
    // read of the staging buffers (its compaction).  Calls with distinct
    // staging buffers never share an event, so they may run concurrently from
    // any threads; the set is checked out for the duration of the call.
    EventSet *ev = nullptr;
    int rc0 = checkout_events(k_dev, s.n_layers + 1, &ev);
    if (rc0) return rc0;
    struct Release {
        EventSet *e;
        ~Release() { checkin_events(e); }
    } release{ev};
    const size_t es = s.dtype == KVC_F32 ? 4 : 2;
    const size_t q_layer = (size_t)s.n_q_heads * s.window * s.head_dim * es;
    const size_t k_layer = (size_t)s.n_kv_heads * s.seq_len * s.head_dim * es;
    // 0. last_done marks the end of the previous call's last read of these
    // staging buffers (its compaction); this call's copies start after it --
    // and only after it, so whatever the caller enqueued since (reading the
    // outputs back) overlaps with the next prompt's copies.  Waiting on an
    // event that was never recorded returns at once.
    cudaError_t e = cudaStreamWaitEvent(copy_stream, ev->last_done, 0);
    // 1. the copy stream moves Q, then K layer by layer, marking each layer
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(q_dev, q_host, q_layer * s.n_layers, cudaMemcpyHostToDevice,
                            copy_stream);
    if (e == cudaSuccess) e = cudaEventRecord(ev->layer[0], copy_stream);
    for (int l = 0; l < s.n_layers && e == cudaSuccess; ++l) {
        e = cudaMemcpyAsync(static_cast<char *>(k_dev) + l * k_layer,
                            static_cast<const char *>(k_host) + l * k_layer, k_layer,
                            cudaMemcpyHostToDevice, copy_stream);
        if (e == cudaSuccess) e = cudaEventRecord(ev->layer[l + 1], copy_stream);
    }
    if (e != cudaSuccess) return fail(KVC_ERR_CUDA, "kvc_compress_host: copy: %s", cudaGetErrorString(e));
    // 2. each layer is scored as soon as its keys have landed
    kvc_shape s1 = s;
    s1.n_layers = 1;
    e = cudaStreamWaitEvent(stream, ev->layer[0], 0);
    for (int l = 0; l < s.n_layers; ++l) {
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ev->layer[l + 1], 0);
        if (e != cudaSuccess) return fail(KVC_ERR_CUDA, "kvc_compress_host: %s", cudaGetErrorString(e));
        const int rc = kvc_score(&s1, static_cast<const char *>(q_dev) + l * q_layer,
                                 static_cast<const char *>(k_dev) + l * k_layer,
                                 scores + (size_t)l * s.n_kv_heads * s.seq_len, ws, ws_bytes, stream);
        if (rc) return rc;
    }
    // 3. budgets, selection and compaction over all layers
    int rc = kvc_mba_budget(&s, scores, mass_num, mass_den, total_budget, layer_floor, mba, budget,
                            ws, ws_bytes, stream);
    if (rc) return rc;
    rc = kvc_topk_select(&s, scores, budget, k_max, idx, ws, ws_bytes, stream);
    if (rc) return rc;
    rc = kvc_compact(&s, k_dev, v_dev, idx, budget, k_max, k_out, v_out, out_rows, ws, ws_bytes,
                     stream);
    if (rc) return rc;
    e = cudaEventRecord(ev->last_done, stream);
    if (e != cudaSuccess) return fail(KVC_ERR_CUDA, "kvc_compress_host: %s", cudaGetErrorString(e));
    return KVC_OK;
}

int kvc_score_keyformer(const kvc_shape *shape, const void *q_obs, const void *k, uint64_t seed,
                        double tau, float *scores, void *ws, size_t ws_bytes, cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_score_keyformer");
    g_err[0] = 0;
    if (!shape_ok(shape, "kvc_score_keyformer")) return KVC_ERR_INVALID_ARG;
    if (!q_obs || !k || !scores) return fail(KVC_ERR_INVALID_ARG, "kvc_score_keyformer: NULL tensor");
    if (!(tau > 0.0) || tau > 1e30)
        return fail(KVC_ERR_INVALID_ARG, "kvc_score_keyformer: tau must be in (0, 1e30]");
    const kvc_shape &s = *shape;
    const WsLayout w = ws_layout(s);
    if (!ws_ok(ws, ws_bytes, w.total, "kvc_score_keyformer")) return KVC_ERR_WORKSPACE;
    const int choice = score_impl_choice();
    if (choice < 0)
        return fail(KVC_ERR_INVALID_ARG, "kvc_score_keyformer: KVC_SCORE_IMPL must be auto, simt or tc");
    const bool can_tc = tc_eligible(s);
    if (choice == 2 && !can_tc)
        return fail(KVC_ERR_UNSUPPORTED, "kvc_score_keyformer: tensor-core path needs bf16, head_dim "
                                         "64/128, G*W <= 512 and an sm_100-family device");
    const bool tc = can_tc && choice != 1;
    if (tc && !aligned16(q_obs)) return fail(KVC_ERR_INVALID_ARG, "kvc_score_keyformer: q_obs must be 16-byte aligned");
    if (tc && !aligned16(k)) return fail(KVC_ERR_INVALID_ARG, "kvc_score_keyformer: k must be 16-byte aligned");
    const ScoreSplit sp = make_split(s, tc);
    ScoreArgs a;
    a.q = q_obs;
    a.k = k;
    a.scores = scores;
    a.partial = reinterpret_cast<float2 *>(static_cast<char *>(ws) + w.partial_off);
    a.neg_bias = reinterpret_cast<float *>(static_cast<char *>(ws) + w.bias_off);
    a.status = status_word(ws);
    stats_forget(ws);   // the noisy statistics replace the plain ones
    return tc ? launch_score_tc_keyformer(s, sp, a, seed, tau, stream)
              : launch_score_keyformer(s, sp, a, seed, tau, stream);
}

int kvc_mba_budget(const kvc_shape *shape, const float *scores, uint32_t mass_num, uint32_t mass_den,
                   int64_t total_budget, int32_t layer_floor, int32_t *mba, int32_t *budget, void *ws,
                   size_t ws_bytes, cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_mba_budget");
    g_err[0] = 0;
    if (!shape_ok(shape, "kvc_mba_budget")) return KVC_ERR_INVALID_ARG;
    const kvc_shape &s = *shape;
    if (!scores || !mba || !budget) return fail(KVC_ERR_INVALID_ARG, "kvc_mba_budget: NULL tensor");
    if (mass_den == 0 || mass_num > mass_den)
        return fail(KVC_ERR_INVALID_ARG, "kvc_mba_budget: need 0 < mass_den and mass_num <= mass_den");
    const int64_t P = (int64_t)s.seq_len - s.window;
    if (layer_floor < 0 || layer_floor > P)
        return fail(KVC_ERR_INVALID_ARG, "kvc_mba_budget: layer_floor must be in [0, T-W]");
    if (total_budget < (int64_t)s.n_layers * layer_floor)
        return fail(KVC_ERR_INVALID_ARG, "kvc_mba_budget: total_budget below n_layers * layer_floor");
    if (!ws_ok(ws, ws_bytes, kWsHeader, "kvc_mba_budget")) return KVC_ERR_WORKSPACE;
    return launch_mba_budget(s, scores, mass_num, mass_den, total_budget, layer_floor, mba, budget,
                             mba_done_word(ws), status_word(ws), stream);
}

int kvc_topk_select(const kvc_shape *shape, const float *scores, const int32_t *budget, int32_t k_max,
                    int32_t *idx, void *ws, size_t ws_bytes, cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_topk_select");
    g_err[0] = 0;
    if (!shape_ok(shape, "kvc_topk_select")) return KVC_ERR_INVALID_ARG;
    if (!scores || !budget || !idx) return fail(KVC_ERR_INVALID_ARG, "kvc_topk_select: NULL tensor");
    if (k_max < 1) return fail(KVC_ERR_INVALID_ARG, "kvc_topk_select: k_max must be >= 1");
    if (!ws_ok(ws, ws_bytes, kWsHeader, "kvc_topk_select")) return KVC_ERR_WORKSPACE;
    return launch_topk(*shape, scores, budget, 0, k_max, idx, status_word(ws), stream);
}

int kvc_head_budget(const kvc_shape *shape, const int32_t *mba, const int32_t *budget,
                    int32_t *head_budget, void *ws, size_t ws_bytes, cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_head_budget");
    g_err[0] = 0;
    if (!shape_ok(shape, "kvc_head_budget")) return KVC_ERR_INVALID_ARG;
    if (!mba || !budget || !head_budget) return fail(KVC_ERR_INVALID_ARG, "kvc_head_budget: NULL tensor");
    if (!ws_ok(ws, ws_bytes, kWsHeader, "kvc_head_budget")) return KVC_ERR_WORKSPACE;
    return launch_head_budget(*shape, mba, budget, head_budget, stream);
}

int kvc_topk_select_heads(const kvc_shape *shape, const float *scores, const int32_t *head_budget,
                          int32_t k_max, int32_t *idx, void *ws, size_t ws_bytes,
                          cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_topk_select_heads");
    g_err[0] = 0;
    if (!shape_ok(shape, "kvc_topk_select_heads")) return KVC_ERR_INVALID_ARG;
    if (!scores || !head_budget || !idx)
        return fail(KVC_ERR_INVALID_ARG, "kvc_topk_select_heads: NULL tensor");
    if (k_max < 1) return fail(KVC_ERR_INVALID_ARG, "kvc_topk_select_heads: k_max must be >= 1");
    if (!ws_ok(ws, ws_bytes, kWsHeader, "kvc_topk_select_heads")) return KVC_ERR_WORKSPACE;
    return launch_topk(*shape, scores, head_budget, 1, k_max, idx, status_word(ws), stream);
}

int kvc_threshold_select(const kvc_shape *shape, const float *scores, float tau, int32_t k_max,
                         int32_t *idx, int32_t *counts, void *ws, size_t ws_bytes,
                         cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_threshold_select");
    g_err[0] = 0;
    if (!shape_ok(shape, "kvc_threshold_select")) return KVC_ERR_INVALID_ARG;
    if (!scores || !idx || !counts)
        return fail(KVC_ERR_INVALID_ARG, "kvc_threshold_select: NULL tensor");
    if (k_max < 1) return fail(KVC_ERR_INVALID_ARG, "kvc_threshold_select: k_max must be >= 1");
    if (!(tau == tau)) return fail(KVC_ERR_INVALID_ARG, "kvc_threshold_select: tau is NaN");
    if (!ws_ok(ws, ws_bytes, kWsHeader, "kvc_threshold_select")) return KVC_ERR_WORKSPACE;
    return launch_threshold(*shape, scores, tau, k_max, idx, counts, status_word(ws), stream);
}

int kvc_compact_heads(const kvc_shape *shape, const void *k, const void *v, const int32_t *idx,
                      const int32_t *counts, int32_t k_max, void *k_out, void *v_out,
                      int64_t out_rows, void *ws, size_t ws_bytes, cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_compact_heads");
    g_err[0] = 0;
    if (!shape_ok(shape, "kvc_compact_heads")) return KVC_ERR_INVALID_ARG;
    if (!k || !v || !idx || !counts || !k_out || !v_out)
        return fail(KVC_ERR_INVALID_ARG, "kvc_compact_heads: NULL tensor");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_out) || !aligned16(v_out))
        return fail(KVC_ERR_INVALID_ARG, "kvc_compact_heads: tensors must be 16-byte aligned");
    if (k_max < 1 || out_rows < 0)
        return fail(KVC_ERR_INVALID_ARG, "kvc_compact_heads: bad k_max/out_rows");
    if (!ws_ok(ws, ws_bytes, kWsHeader, "kvc_compact_heads")) return KVC_ERR_WORKSPACE;
    return launch_compact(*shape, k, v, idx, counts, 1, k_max, k_out, v_out, out_rows,
                          status_word(ws), stream);
}

int kvc_pool_scores(const kvc_shape *shape, const float *scores, int32_t kernel, int32_t mode,
                    float *pooled, void *ws, size_t ws_bytes, cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_pool_scores");
    g_err[0] = 0;
    if (!shape_ok(shape, "kvc_pool_scores")) return KVC_ERR_INVALID_ARG;
    if (!scores || !pooled) return fail(KVC_ERR_INVALID_ARG, "kvc_pool_scores: NULL tensor");
    if (scores == pooled)
        return fail(KVC_ERR_INVALID_ARG, "kvc_pool_scores: pooled must not alias scores");
    if (kernel < 1 || (kernel & 1) == 0)
        return fail(KVC_ERR_INVALID_ARG, "kvc_pool_scores: kernel must be odd and >= 1");
    if (mode != 0 && mode != 1)
        return fail(KVC_ERR_INVALID_ARG, "kvc_pool_scores: mode must be 0 (average) or 1 (max)");
    if (!ws_ok(ws, ws_bytes, kWsHeader, "kvc_pool_scores")) return KVC_ERR_WORKSPACE;
    return launch_pool(*shape, scores, kernel, mode, pooled, stream);
}

int kvc_compact(const kvc_shape *shape, const void *k, const void *v, const int32_t *idx,
                const int32_t *budget, int32_t k_max, void *k_out, void *v_out, int64_t out_rows,
                void *ws, size_t ws_bytes, cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_compact");
    g_err[0] = 0;
    if (!shape_ok(shape, "kvc_compact")) return KVC_ERR_INVALID_ARG;
    if (!k || !v || !idx || !budget || !k_out || !v_out)
        return fail(KVC_ERR_INVALID_ARG, "kvc_compact: NULL tensor");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_out) || !aligned16(v_out))
        return fail(KVC_ERR_INVALID_ARG, "kvc_compact: tensors must be 16-byte aligned");
    if (k_max < 1 || out_rows < 0) return fail(KVC_ERR_INVALID_ARG, "kvc_compact: bad k_max/out_rows");
    if (!ws_ok(ws, ws_bytes, kWsHeader, "kvc_compact")) return KVC_ERR_WORKSPACE;
    return launch_compact(*shape, k, v, idx, budget, 0, k_max, k_out, v_out, out_rows, status_word(ws),
                          stream);
}

int32_t kvc_keep_channels(double lambda, int32_t head_dim) {
    if (!(lambda >= 0.0 && lambda < 1.0) || head_dim < 1) return 0;
    return (int32_t)std::floor((1.0 - lambda) * (double)head_dim);
}

int kvc_channel_prune(const kvc_shape *shape, const void *k_out, const int32_t *budget, double lambda,
                      int32_t *chan, void *k_pruned, int64_t pruned_elems, void *ws, size_t ws_bytes,
                      cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_channel_prune");
    g_err[0] = 0;
    if (!shape_ok(shape, "kvc_channel_prune")) return KVC_ERR_INVALID_ARG;
    if (!k_out || !budget || !chan || !k_pruned)
        return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune: NULL tensor");
    const int32_t keep = kvc_keep_channels(lambda, shape->head_dim);
    if (keep < 1) return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune: lambda keeps no channel");
    if (pruned_elems < 0) return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune: bad pruned_elems");
    if (!ws_ok(ws, ws_bytes, kWsHeader, "kvc_channel_prune")) return KVC_ERR_WORKSPACE;
    return launch_channel_prune(*shape, nullptr, k_out, budget, keep, chan, k_pruned, pruned_elems,
                                status_word(ws), stream);
}

int kvc_channel_prune_value(const kvc_shape *shape, const void *q_obs, const void *k,
                            const void *v, const void *v_out, const int32_t *budget, double lambda,
                            float *value_scores, int32_t *chan, void *v_pruned,
                            int64_t pruned_elems, void *ws, size_t ws_bytes, cudaStream_t stream) {
    return kvc_channel_prune_value_ex(shape, q_obs, k, v, v_out, budget, lambda, value_scores, chan,
                                      v_pruned, pruned_elems, 0u, ws, ws_bytes, stream);
}

int kvc_channel_prune_value_ex(const kvc_shape *shape, const void *q_obs, const void *k,
                               const void *v, const void *v_out, const int32_t *budget,
                               double lambda, float *value_scores, int32_t *chan, void *v_pruned,
                               int64_t pruned_elems, uint32_t flags, void *ws, size_t ws_bytes,
                               cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_channel_prune_value");
    g_err[0] = 0;
    if (!shape_ok(shape, "kvc_channel_prune_value")) return KVC_ERR_INVALID_ARG;
    const kvc_shape &s = *shape;
    if (!q_obs || !k || !v || !v_out || !budget || !chan || !v_pruned)
        return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune_value: NULL tensor");
    if (!aligned16(q_obs) || !aligned16(k) || !aligned16(v))
        return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune_value: q_obs, k and v must be 16-byte aligned");
    const int32_t keep = kvc_keep_channels(lambda, s.head_dim);
    if (keep < 1) return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune_value: lambda keeps no channel");
    if (pruned_elems < 0) return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune_value: bad pruned_elems");
    if (flags & ~KVC_VALUE_REUSE_SCORE_STATS)
        return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune_value_ex: unknown flags %#x", flags);
    const WsLayout w = ws_layout(s);
    if (!ws_ok(ws, ws_bytes, w.total, "kvc_channel_prune_value")) return KVC_ERR_WORKSPACE;
    const int choice = score_impl_choice();
    if (choice < 0)
        return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune_value: KVC_SCORE_IMPL must be auto, simt or tc");
    const bool can_tc = tc_eligible(s);
    if (choice == 2 && !can_tc)
        return fail(KVC_ERR_UNSUPPORTED, "kvc_channel_prune_value: tensor-core path needs bf16, "
                                         "head_dim 64/128, G*W <= 512 and an sm_100-family device");
    const bool tc = can_tc && choice != 1;
    const ScoreSplit sp = make_split(s, tc);
    char *base = static_cast<char *>(ws);
    // 1. the window rows' softmax normalisers (the score pass's first half),
    // or those the last kvc_score over the same shape, q_obs and k left here
    ScoreArgs a;
    a.q = q_obs;
    a.k = k;
    a.scores = nullptr;
    a.partial = reinterpret_cast<float2 *>(base + w.partial_off);
    a.neg_bias = reinterpret_cast<float *>(base + w.bias_off);
    a.status = status_word(ws);
    a.stats_only = true;
    int rc = KVC_OK;
    if (flags & KVC_VALUE_REUSE_SCORE_STATS) {
        if (!stats_match(ws, s, q_obs, k, tc))
            return fail(KVC_ERR_INVALID_ARG,
                        "kvc_channel_prune_value_ex: no kvc_score over this shape, q_obs and k is "
                        "recorded for this workspace");
    } else {
        rc = tc ? launch_score_tc(s, sp, a, stream) : launch_score_simt(s, sp, a, stream);
        if (rc) {
            stats_forget(ws);
            return rc;
        }
        stats_record(ws, s, q_obs, k, tc);
    }
    // 2. per-channel squared norms of the window rows' attention output
    float *sv = value_scores ? value_scores : reinterpret_cast<float *>(base + w.vscore_off);
    rc = launch_value_scores(s, sp, q_obs, k, v, a.neg_bias,
                             reinterpret_cast<float *>(base + w.vpart_off), sv,
                             tc && value_tc_eligible(s), status_word(ws), stream);
    if (rc) return rc;
    // 3. keep the top channels and copy them out of the kept prefix rows
    return launch_channel_prune(s, nullptr, v_out, budget, keep, chan, v_pruned, pruned_elems,
                                status_word(ws), stream, sv);
}

int kvc_channel_prune_query(const kvc_shape *shape, const void *q_obs, const void *k_out,
                            const int32_t *budget, double lambda, int32_t *chan, void *k_pruned,
                            int64_t pruned_elems, void *ws, size_t ws_bytes, cudaStream_t stream) {
    NvtxRange nvtx_range("kvc_channel_prune_query");
    g_err[0] = 0;
    if (!shape_ok(shape, "kvc_channel_prune_query")) return KVC_ERR_INVALID_ARG;
    if (!q_obs || !k_out || !budget || !chan || !k_pruned)
        return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune_query: NULL tensor");
    const int32_t keep = kvc_keep_channels(lambda, shape->head_dim);
    if (keep < 1) return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune_query: lambda keeps no channel");
    if (pruned_elems < 0)
        return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune_query: bad pruned_elems");
    if (!ws_ok(ws, ws_bytes, kWsHeader, "kvc_channel_prune_query")) return KVC_ERR_WORKSPACE;
    return launch_channel_prune(*shape, q_obs, k_out, budget, keep, chan, k_pruned, pruned_elems,
                                status_word(ws), stream);
}

const char *kvc_status_string(int status) {
    switch (status) {
        case KVC_OK: return "ok";
        case KVC_ERR_INVALID_ARG: return "invalid argument";
        case KVC_ERR_UNSUPPORTED: return "unsupported";
        case KVC_ERR_CUDA: return "CUDA error";
        case KVC_ERR_TIMEOUT: return "device wait timed out";
        case KVC_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

const char *kvc_last_error(void) { return g_err; }

}  // extern "C"
