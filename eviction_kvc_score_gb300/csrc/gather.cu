// gather.cu -- K/V compaction and ThinK key-channel pruning.
//
// Compaction (blog post "ZigZagKV, KVCache 80% compression near-lossless",
// section "SnapKV": the kept tokens are the top-K plus every token of the
// last window): for head (l,k) the output block holds the n_l kept prefix
// rows in ascending position order, then the W window rows.  The copy is
// pure data movement: each thread moves 16-byte vectors, consecutive threads
// write consecutive addresses, reads are whole rows gathered by index.  With
// per-head counts (per-head budgets or threshold selection) head (l,k) keeps
// its own n_{l,k} rows and the heads follow each other in (l, k) order.
//
// ThinK ("ThinK: Thinner Key Cache by Query-Driven Pruning", "Magnitude-based
// pruning", "Implementation of THINK"): per head, M_d = ||K[:, d]||_2^2 over
// the kept prefix rows, keep the floor((1-lambda) D) largest channels (ties to
// the lower d), copy them for the prefix rows; window rows stay full width.
// Sums of squares run in a float-float pair (error-free products via FMA and
// TwoSum additions), about 44 significant bits, so the channel order matches
// an fp64 sum except for channels equal to within ~1e-13.
#include <cooperative_groups.h>

#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int kCopyThreads = 256;
constexpr int kRowsPerBlock = 64;

__device__ __forceinline__ int64_t kept(int32_t b, int P) {
    return b < 0 ? 0 : (b > P ? P : b);
}

// Row offset of layer l in the packed output (in rows), computed from the
// device budgets.
__device__ __forceinline__ int64_t layer_row_offset(const int32_t *budget, int l, int Hkv, int P,
                                                    int W) {
    int64_t off = 0;
    for (int i = 0; i < l; ++i) off += (int64_t)Hkv * (kept(budget[i], P) + W);
    return off;
}

template <typename V>
__global__ void __launch_bounds__(kCopyThreads)
    compact_kernel(const V *__restrict__ k, const V *__restrict__ v, const int32_t *__restrict__ idx,
                   const int32_t *__restrict__ budget, int per_head, int T, int W, int Hkv,
                   int k_max, int vec_per_row, V *__restrict__ k_out, V *__restrict__ v_out,
                   int64_t out_rows, uint32_t *status) {
    __shared__ int64_t s_row0;
    __shared__ int s_n;
    const int head = blockIdx.x;
    const int l = head / Hkv, h = head % Hkv;
    const int P = T - W;
    if (threadIdx.x == 0) {
        if (per_head) {
            // budget holds one count per head; heads follow each other
            int64_t off = 0;
            for (int u = 0; u < head; ++u) off += min(kept(budget[u], P), (int64_t)k_max) + W;
            s_n = (int)min(kept(budget[head], P), (int64_t)k_max);
            s_row0 = off;
        } else {
            int64_t n = kept(budget[l], P);
            if (n > k_max) n = k_max;   // reported by the top-K step
            s_n = (int)n;
            s_row0 = layer_row_offset(budget, l, Hkv, P, W) + (int64_t)h * (kept(budget[l], P) + W);
        }
    }
    __syncthreads();
    const int n = s_n;
    const int64_t row0 = s_row0;
    const int rows = n + W;
    const int32_t *sel = idx + (int64_t)head * k_max;
    const V *ks = k + (int64_t)head * T * vec_per_row;
    const V *vs = v + (int64_t)head * T * vec_per_row;
    for (int rb = blockIdx.y * kRowsPerBlock; rb < rows; rb += gridDim.y * kRowsPerBlock) {
        const int rend = min(rows, rb + kRowsPerBlock);
        const int total = (rend - rb) * vec_per_row;
        for (int i = threadIdx.x; i < total; i += kCopyThreads) {
            const int r = rb + i / vec_per_row;
            const int e = i % vec_per_row;
            const int64_t orow = row0 + r;
            if (orow >= out_rows) {
                set_status(status, KVC_DEV_OUT_CAPACITY);
                continue;
            }
            const int t = r < n ? sel[r] : P + (r - n);
            if (t < 0 || t >= T) {
                set_status(status, KVC_DEV_BAD_BUDGET);
                continue;
            }
            // kept prefix positions strictly ascending and inside the prefix
            if (kDebugBounds && e == 0 && r < n && (t >= P || (r > 0 && sel[r - 1] >= t)))
                set_status(status, KVC_DEV_INVARIANT);
            k_out[orow * vec_per_row + e] = ks[(int64_t)t * vec_per_row + e];
            v_out[orow * vec_per_row + e] = vs[(int64_t)t * vec_per_row + e];
        }
    }
}

// ------------------------------------------------------------------ ThinK
struct FF {   // unevaluated sum hi + lo
    float hi, lo;
};

__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

__device__ __forceinline__ FF ff_add(FF a, FF b) {
    float s, e;
    two_sum(a.hi, b.hi, s, e);
    e += a.lo + b.lo;
    FF r;
    two_sum(s, e, r.hi, r.lo);
    return r;
}

__device__ __forceinline__ FF ff_add_sq(FF a, float x) {
    const float p = x * x;
    const float pe = fmaf(x, x, -p);   // exact product error
    float s, e;
    two_sum(a.hi, p, s, e);
    e += a.lo + pe;
    FF r;
    two_sum(s, e, r.hi, r.lo);
    return r;
}

template <typename T>
__device__ __forceinline__ float ld_f(const T *p, int64_t i);
template <>
__device__ __forceinline__ float ld_f<float>(const float *p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}

constexpr int kPruneThreads = 512;
constexpr int kPruneWarps = kPruneThreads / 32;
constexpr int kPruneCluster = 8;   // CTAs per head, one cluster

// x^2 added to a float-float sum.  A bf16 value has 8 significant bits, so
// its square is exact in fp32; an fp32 square carries its FMA-recovered
// rounding error.
template <typename T>
__device__ __forceinline__ FF ff_add_sq_t(FF a, float x) {
    if constexpr (sizeof(T) == 2) {
        float s, e;
        two_sum(a.hi, x * x, s, e);
        e += a.lo;
        FF r;
        two_sum(s, e, r.hi, r.lo);
        return r;
    } else {
        return ff_add_sq(a, x);
    }
}

// Per-channel float-float sums of squares over rows [lo, hi) of the
// row-major [rows][D] block starting at row first_row of base: warp w takes
// rows lo + w, lo + w + 16, ...; lane l owns channels l + 32 k, so each load
// instruction of a warp reads consecutive elements of one row.  The warps'
// partial sums are added in warp order (a fixed order: every CTA of a head
// gets the same bits for the same slice).
template <typename T, int CPL>
__device__ void slice_sums(const T *__restrict__ base, int64_t first_row, int lo, int hi, int D,
                           FF *wpart, FF *out) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    FF a[CPL];
#pragma unroll
    for (int k = 0; k < CPL; ++k) a[k] = {0.f, 0.f};
    int r = lo + warp;
    // four rows' loads in flight before their (dependent) sums: the warp's
    // rows are few and HBM latency, not bandwidth, would set the pace
    constexpr int kRowsInFlight = 4;
    for (; r + (kRowsInFlight - 1) * kPruneWarps < hi; r += kRowsInFlight * kPruneWarps) {
        float x[kRowsInFlight][CPL];
#pragma unroll
        for (int i = 0; i < kRowsInFlight; ++i) {
            const T *ri = base + (first_row + r + (int64_t)i * kPruneWarps) * D;
#pragma unroll
            for (int k = 0; k < CPL; ++k) {
                const int c = lane + 32 * k;
                x[i][k] = c < D ? ld_f(ri, c) : 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < kRowsInFlight; ++i)
#pragma unroll
            for (int k = 0; k < CPL; ++k) a[k] = ff_add_sq_t<T>(a[k], x[i][k]);
    }
    for (; r < hi; r += kPruneWarps) {
        const T *r0 = base + (first_row + r) * D;
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
            const int c = lane + 32 * k;
            if (c < D) a[k] = ff_add_sq_t<T>(a[k], ld_f(r0, c));
        }
    }
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const int c = lane + 32 * k;
        if (c < D) wpart[warp * D + c] = a[k];
    }
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += kPruneThreads) {
        FF t = wpart[c];
        for (int w = 1; w < kPruneWarps; ++w) t = ff_add(t, wpart[w * D + c]);
        out[c] = t;
    }
    __syncthreads();
}

// One cluster of kPruneCluster CTAs per head: CTA `rank` owns a contiguous
// slice of the head's kept prefix rows (and of its window-query rows for the
// query-driven criterion).  Each CTA forms float-float per-channel sums of
// squares over its slice; after a cluster barrier every CTA adds the slices'
// sums in rank order from distributed shared memory -- the same fixed order
// in every CTA, so all of them rank the channels identically -- and copies
// the chosen channels of its own rows: a warp per row, lane l writing output
// positions l + 32 k from source channels fixed for the head (coalesced
// stores, no per-element index arithmetic).  CPL = channels per lane
// (D <= 32 CPL).
template <typename T, int CPL>
__global__ void __launch_bounds__(kPruneThreads)
    channel_prune_kernel(const T *__restrict__ k_out, const T *__restrict__ q, int Hq,
                         const int32_t *__restrict__ budget, int T_len, int W, int Hkv, int D,
                         int keep, int32_t *__restrict__ chan, T *__restrict__ k_pruned,
                         int64_t pruned_elems, uint32_t *status, const float *__restrict__ given) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ FF wpart[kPruneWarps * 32 * CPL];
    __shared__ FF slice_k[32 * CPL], slice_q[32 * CPL];
    __shared__ unsigned long long m[32 * CPL];   // channel scores as ordered keys
    __shared__ int sel[32 * CPL];
    __shared__ int flag[32 * CPL];
    __shared__ int64_t s_row0, s_o0;
    __shared__ int s_n;
    const int rank = (int)cluster.block_rank();
    const int head = blockIdx.x / kPruneCluster;
    const int l = head / Hkv, h = head % Hkv;
    const int P = T_len - W;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    if (warp == 0) {
        // kept prefix rows of the layers before l, summed by the warp (the
        // loads in parallel, not one dependent load per layer)
        int64_t o = 0;
        for (int i = lane; i < l; i += 32) o += kept(budget[i], P);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) o += __shfl_xor_sync(0xffffffffu, o, off);
        if (lane == 0) {
            const int64_t n = kept(budget[l], P);
            s_n = (int)n;
            // each earlier layer holds Hkv heads of (kept + W) rows
            s_row0 = (int64_t)Hkv * (o + (int64_t)l * W) + (int64_t)h * (n + W);
            s_o0 = ((int64_t)Hkv * o + (int64_t)h * n) * keep;
        }
    }
    __syncthreads();
    const int n = s_n;
    const int64_t row0 = s_row0;
    const int r_lo = (int)((int64_t)n * rank / kPruneCluster);
    const int r_hi = (int)((int64_t)n * (rank + 1) / kPruneCluster);

    // 1. this CTA's slice: per-channel sums of squares of its rows
    if (given == nullptr) slice_sums<T, CPL>(k_out, row0, r_lo, r_hi, D, wpart, slice_k);
    if (given == nullptr && q != nullptr) {
        // query-driven criterion: the W window rows of each of the head's G
        // query heads, split over the cluster like the key rows
        const int G = Hq / Hkv;
        const int qrows = G * W;
        slice_sums<T, CPL>(q, ((int64_t)l * Hq + (int64_t)h * G) * W,
                           (int)((int64_t)qrows * rank / kPruneCluster),
                           (int)((int64_t)qrows * (rank + 1) / kPruneCluster), D, wpart, slice_q);
    }
    cluster.sync();

    // 2. whole-head sums in rank order, then rank by (score desc, d asc).
    // The scores are non-negative doubles, whose bit patterns order like the
    // values as 64-bit integers: the D x D comparisons run on integer units
    // (this part's FP64 rate is a small fraction of its FP32 rate).
    if (tid < D && given != nullptr) {
        const double mg = (double)given[(int64_t)head * D + tid];   // THINKV: scores supplied
        m[tid] = (unsigned long long)__double_as_longlong(mg > 0.0 ? mg : 0.0);
    } else if (tid < D) {
        FF tk = {0.f, 0.f}, tq = {0.f, 0.f};
        for (int rr = 0; rr < kPruneCluster; ++rr) {
            tk = ff_add(tk, cluster.map_shared_rank(slice_k, rr)[tid]);
            if (q != nullptr) tq = ff_add(tq, cluster.map_shared_rank(slice_q, rr)[tid]);
        }
        double mk = (double)tk.hi + (double)tk.lo;
        if (q != nullptr) mk *= (double)tq.hi + (double)tq.lo;
        m[tid] = (unsigned long long)__double_as_longlong(mk > 0.0 ? mk : 0.0);
    }
    __syncthreads();
    if (tid < D) {
        const unsigned long long mine = m[tid];
        int rk = 0;
        for (int o = 0; o < D; ++o) rk += (m[o] > mine) || (m[o] == mine && o < tid);
        flag[tid] = rk < keep;
    }
    __syncthreads();
    if (tid < D && flag[tid]) {
        int pos = 0;
        for (int o = 0; o < tid; ++o) pos += flag[o];
        sel[pos] = tid;
        if (rank == 0) chan[(int64_t)head * keep + pos] = tid;
    }
    // no CTA may leave while another still reads its slice sums
    cluster.sync();
    if (kDebugBounds && rank == 0 && tid < keep &&
        (sel[tid] < 0 || sel[tid] >= D || (tid > 0 && sel[tid - 1] >= sel[tid])))
        set_status(status, KVC_DEV_INVARIANT);   // keep channels, strictly ascending

    // 3. copy the kept channels of this CTA's rows: warp per row
    int src[CPL];
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const int j = lane + 32 * k;
        src[k] = j < keep ? sel[j] : -1;
    }
    if (s_o0 + (int64_t)r_hi * keep > pruned_elems && tid == 0)
        set_status(status, KVC_DEV_OUT_CAPACITY);   // output too small: copy what fits
#pragma unroll 4
    for (int r = r_lo + warp; r < r_hi; r += kPruneWarps) {
        const T *s_row = k_out + (row0 + r) * D;
        const int64_t o = s_o0 + (int64_t)r * keep;
        T *d_row = k_pruned + o;
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
            const int j = lane + 32 * k;
            if (src[k] >= 0 && o + j < pruned_elems) d_row[j] = s_row[src[k]];
        }
    }
}

template <typename T>
cudaError_t launch_prune_t(const kvc_shape &s, const void *q, const void *k_out,
                           const int32_t *budget, int32_t keep, int32_t *chan, void *k_pruned,
                           int64_t pruned_elems, uint32_t *status, cudaStream_t st,
                           const float *given) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(s.n_layers * s.n_kv_heads * kPruneCluster));
    cfg.blockDim = dim3(kPruneThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPruneCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto go = [&](auto kernel) {
        return cudaLaunchKernelEx(&cfg, kernel, (const T *)k_out, (const T *)q, s.n_q_heads, budget,
                                  s.seq_len, s.window, s.n_kv_heads, s.head_dim, (int)keep, chan,
                                  (T *)k_pruned, pruned_elems, status, given);
    };
    // channels per lane of the sums and the copy
    if (s.head_dim <= 64) return go(channel_prune_kernel<T, 2>);
    if (s.head_dim <= 128) return go(channel_prune_kernel<T, 4>);
    return go(channel_prune_kernel<T, 8>);
}

}  // namespace

int launch_compact(const kvc_shape &s, const void *k, const void *v, const int32_t *idx,
                   const int32_t *budget, int per_head, int32_t k_max, void *k_out, void *v_out,
                   int64_t out_rows, uint32_t *status, cudaStream_t st) {
    const size_t es = s.dtype == KVC_F32 ? 4 : 2;
    const size_t row_bytes = es * (size_t)s.head_dim;
    const int heads = s.n_layers * s.n_kv_heads;
    const int max_rows = k_max + s.window;
    dim3 grid(heads, (unsigned)min(32, (max_rows + kRowsPerBlock - 1) / kRowsPerBlock));
    if (row_bytes % 16 == 0) {
        compact_kernel<uint4><<<grid, kCopyThreads, 0, st>>>(
            (const uint4 *)k, (const uint4 *)v, idx, budget, per_head, s.seq_len, s.window,
            s.n_kv_heads, k_max, (int)(row_bytes / 16), (uint4 *)k_out, (uint4 *)v_out, out_rows,
            status);
    } else if (row_bytes % 4 == 0) {
        compact_kernel<uint32_t><<<grid, kCopyThreads, 0, st>>>(
            (const uint32_t *)k, (const uint32_t *)v, idx, budget, per_head, s.seq_len, s.window,
            s.n_kv_heads, k_max, (int)(row_bytes / 4), (uint32_t *)k_out, (uint32_t *)v_out,
            out_rows, status);
    } else {
        compact_kernel<uint16_t><<<grid, kCopyThreads, 0, st>>>(
            (const uint16_t *)k, (const uint16_t *)v, idx, budget, per_head, s.seq_len, s.window,
            s.n_kv_heads, k_max, (int)(row_bytes / 2), (uint16_t *)k_out, (uint16_t *)v_out,
            out_rows, status);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_compact: launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

int launch_channel_prune(const kvc_shape &s, const void *q, const void *k_out, const int32_t *budget,
                         int32_t keep, int32_t *chan, void *k_pruned, int64_t pruned_elems,
                         uint32_t *status, cudaStream_t st, const float *given) {
    if (s.head_dim > 256) {
        set_error("kvc_channel_prune: head_dim above 256 is not supported");
        return KVC_ERR_UNSUPPORTED;
    }
    cudaError_t e0 = s.dtype == KVC_F32
                         ? launch_prune_t<float>(s, q, k_out, budget, keep, chan, k_pruned,
                                                 pruned_elems, status, st, given)
                         : launch_prune_t<__nv_bfloat16>(s, q, k_out, budget, keep, chan, k_pruned,
                                                         pruned_elems, status, st, given);
    if (e0 != cudaSuccess) {
        set_error("kvc_channel_prune: launch failed: %s", cudaGetErrorString(e0));
        return KVC_ERR_CUDA;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_channel_prune: launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

}  // namespace kvc
