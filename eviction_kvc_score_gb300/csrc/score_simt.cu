// score_simt.cu -- observation-window scores on the CUDA cores (fp32 FFMA),
// for fp32 inputs and for bf16 shapes outside the tensor-core kernel's range
// (head_dim other than 64/128, or more than 512 window rows per KV head);
// the merge of pass-1 partial row statistics used by both paths; and the
// optional Keyformer scores ("Keyformer: KV Cache reduction through key
// tokens selection": Gumbel noise on the logits, temperature softmax), the
// same two passes with a counter-based Gumbel draw per (unit, row, key).
//
// Same two-pass definition as score_tc.cu (SnapKV window scoring with
// softmax(q.k / sqrt(D)), causal inside the window, GQA rows averaged), same
// work split over (unit, 128-key tile) pairs and the same partial layout, so
// the merge kernel serves both.
#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int kSimtThreads = 128;
constexpr int kSub = 32;  // keys per shared-memory sub-tile (pass 1) / rows per chunk (pass 2)

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

struct SimtParams {
    int64_t n_tiles, tiles_per_unit;
    int grid, max_slots;
    int T, P, W, D, rows, rows_pad;
    float cs;
    float2 *partial;
    const float *neg_bias;
    float *scores;
    // Keyformer noise (NOISE kernels only): Philox key, log2(e) / tau
    uint32_t key0, key1;
    float noise_scale;
};

// Pass 1: thread = query row; for each 32-key sub-tile held in shared memory
// the thread forms its 32 logits and folds them into an online (max, sum).
template <typename T, bool NOISE>
__global__ void __launch_bounds__(kSimtThreads)
    score_stats_simt(const T *__restrict__ q, const T *__restrict__ k, SimtParams p) {
    extern __shared__ float ks[];                   // [kSub][D]
    const int64_t c = blockIdx.x;
    const int64_t t0 = split_begin(p.n_tiles, p.grid, c), t1 = split_begin(p.n_tiles, p.grid, c + 1);
    const int D = p.D;
    for (int rbase = 0; rbase < p.rows; rbase += kSimtThreads) {
        const int r = rbase + threadIdx.x;
        const bool row_ok = r < p.rows;
        const int w = row_ok ? r % p.W : 0;
        float m_run = -INFINITY, l_run = 0.f;
        for (int64_t t = t0; t < t1; ++t) {
            const int64_t u = t / p.tiles_per_unit;
            const int jt = (int)(t % p.tiles_per_unit);
            if (t == t0 || jt == 0) {
                m_run = -INFINITY;
                l_run = 0.f;
            }
            const T *qr = q + ((u * p.rows) + (row_ok ? r : 0)) * (int64_t)D;
            const T *ku = k + u * (int64_t)p.T * D;
            for (int sub = 0; sub < kTileKeys; sub += kSub) {
                const int j0 = jt * kTileKeys + sub;
                __syncthreads();
                for (int e = threadIdx.x; e < kSub * D; e += kSimtThreads) {
                    const int jj = j0 + e / D;
                    ks[e] = jj < p.T ? to_f(ku[(int64_t)jj * D + e % D]) : 0.f;
                }
                __syncthreads();
                float s[kSub];
#pragma unroll
                for (int i = 0; i < kSub; ++i) s[i] = 0.f;
                for (int d = 0; d < D; ++d) {
                    const float qd = to_f(qr[d]);
#pragma unroll
                    for (int i = 0; i < kSub; ++i) s[i] = fmaf(qd, ks[i * D + d], s[i]);
                }
                const int lim = p.P + w - j0;   // largest visible sub-tile column
                if (NOISE) {
                    // base-2 noisy logits (x / sqrt(D) + zeta) / tau, logits
                    // beyond the causal limit stay out of the max and sum
                    // the sub-tile's keys are whole noise blocks of row r (four
                    // keys each)
                    static_assert(kSub % 4 == 0, "whole Philox blocks per sub-tile");
#pragma unroll
                    for (int i4 = 0; i4 < kSub; i4 += 4) {
                        uint32_t wb[4];
                        philox4((uint32_t)(j0 + i4) >> 2, (uint32_t)r, (uint32_t)u, p.key0,
                                p.key1, wb);
#pragma unroll
                        for (int i = i4; i < i4 + 4; ++i)
                            if (i <= lim && j0 + i < p.T)
                                s[i] = fmaf(gumbel_bits(wb[i & 3]), p.noise_scale, s[i] * p.cs);
                            else
                                s[i] = -INFINITY;
                    }
                    float mxn = -INFINITY;
#pragma unroll
                    for (int i = 0; i < kSub; ++i) mxn = fmaxf(mxn, s[i]);
                    if (mxn > -INFINITY) {
                        const float mnew = fmaxf(m_run, mxn);
                        float sum = 0.f;
#pragma unroll
                        for (int i = 0; i < kSub; ++i) sum += ex2(s[i] - mnew);
                        l_run = l_run * ex2(m_run - mnew) + sum;
                        m_run = mnew;
                    }
                    continue;
                }
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < kSub; ++i)
                    if (i <= lim) mx = fmaxf(mx, s[i]);
                if (mx > -INFINITY) {
                    const float mnew = fmaxf(m_run, mx * p.cs);
                    float sum = 0.f;
#pragma unroll
                    for (int i = 0; i < kSub; ++i)
                        if (i <= lim) sum += ex2(fmaf(s[i], p.cs, -mnew));
                    l_run = l_run * ex2(m_run - mnew) + sum;
                    m_run = mnew;
                }
            }
            const bool last = (t == t1 - 1) || (jt == p.tiles_per_unit - 1);
            if (last && row_ok) {
                const int64_t slot = c - split_cta_of(p.n_tiles, p.grid, u * p.tiles_per_unit);
                p.partial[(u * p.max_slots + slot) * p.rows_pad + r] = make_float2(m_run, l_run);
            }
        }
    }
}

// Pass 2: thread = key; the unit's query rows stream through shared memory
// 32 at a time; each thread sums 2^(x + nb_r) over the rows that see it.
template <typename T, bool NOISE>
__global__ void __launch_bounds__(kSimtThreads)
    score_colmean_simt(const T *__restrict__ q, const T *__restrict__ k, SimtParams p) {
    extern __shared__ float qs[];                   // [kSub][D] then nb[kSub]
    float *nbs = qs + kSub * p.D;
    const int64_t c = blockIdx.x;
    const int64_t t0 = split_begin(p.n_tiles, p.grid, c), t1 = split_begin(p.n_tiles, p.grid, c + 1);
    const int D = p.D;
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t u = t / p.tiles_per_unit;
        const int jt = (int)(t % p.tiles_per_unit);
        const int j = jt * kTileKeys + threadIdx.x;
        const int dj = j - p.P;
        const T *kj = k + (u * (int64_t)p.T + (j < p.T ? j : 0)) * D;
        float acc = 0.f;
        for (int rbase = 0; rbase < p.rows; rbase += kSub) {
            __syncthreads();
            for (int e = threadIdx.x; e < kSub * D; e += kSimtThreads) {
                const int rr = rbase + e / D;
                qs[e] = rr < p.rows ? to_f(q[((u * p.rows) + rr) * (int64_t)D + e % D]) : 0.f;
            }
            for (int e = threadIdx.x; e < kSub; e += kSimtThreads) {
                const int rr = rbase + e;
                nbs[e] = rr < p.rows ? p.neg_bias[u * p.rows_pad + rr] : -INFINITY;
            }
            __syncthreads();
            float s[kSub];
#pragma unroll
            for (int i = 0; i < kSub; ++i) s[i] = 0.f;
            for (int d = 0; d < D; ++d) {
                const float kd = to_f(kj[d]);
#pragma unroll
                for (int i = 0; i < kSub; ++i) s[i] = fmaf(qs[i * D + d], kd, s[i]);
            }
#pragma unroll
            for (int i = 0; i < kSub; ++i) {
                const int rr = rbase + i;
                const bool vis = rr < p.rows && (rr % p.W) >= dj && j < p.T;
                float arg = fmaf(s[i], p.cs, nbs[i]);
                if (NOISE && vis)
                    arg = fmaf(gumbel((uint32_t)u, (uint32_t)rr, (uint32_t)j, p.key0, p.key1),
                               p.noise_scale, arg);
                const float e = ex2(arg);
                acc += vis ? e : 0.f;
            }
        }
        if (j < p.T) p.scores[u * p.T + j] = acc / (float)p.rows;
    }
}

// Merge: nb_r = -(M + log2 sum_s l_s 2^(m_s - M)) over the unit's slots
// (fp32: the few terms are within a factor 2^64 of each other and the result
// needs ~1e-6 relative accuracy; fp64 runs at a small fraction of the fp32
// rate on this GPU); pad rows get -inf so that they contribute nothing in
// pass 2.
__global__ void score_merge(const float2 *__restrict__ partial, float *__restrict__ neg_bias,
                            int64_t n_units, int64_t tiles_per_unit, int64_t n_tiles, int grid,
                            int max_slots, int rows, int rows_pad) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_units * rows_pad) return;
    const int64_t u = i / rows_pad;
    const int r = (int)(i % rows_pad);
    if (r >= rows) {
        neg_bias[i] = -INFINITY;
        return;
    }
    const int64_t first = split_cta_of(n_tiles, grid, u * tiles_per_unit);
    const int64_t last = split_cta_of(n_tiles, grid, u * tiles_per_unit + tiles_per_unit - 1);
    const float2 *pp = partial + u * max_slots * (int64_t)rows_pad + r;
    float m = -INFINITY;
    for (int64_t s = 0; s <= last - first; ++s) m = fmaxf(m, pp[s * rows_pad].x);
    float l = 0.f;
    for (int64_t s = 0; s <= last - first; ++s) {
        const float2 v = pp[s * rows_pad];
        if (v.x > -INFINITY) l += v.y * exp2f(v.x - m);
    }
    neg_bias[i] = -(m + log2f(l));
}

template <typename T, bool NOISE>
int launch_simt_t(const kvc_shape &s, const ScoreSplit &sp, const ScoreArgs &a, cudaStream_t st,
                  uint64_t seed = 0, double tau = 1.0) {
    SimtParams p;
    p.n_tiles = sp.n_tiles;
    p.tiles_per_unit = sp.tiles_per_unit;
    p.grid = sp.grid;
    p.max_slots = sp.max_slots;
    p.T = s.seq_len;
    p.W = s.window;
    p.P = s.seq_len - s.window;
    p.D = s.head_dim;
    p.rows = sp.rows;
    p.rows_pad = sp.rows_pad;
    // Keyformer divides the noisy logits by tau: both the logit scale and
    // the noise scale carry 1/tau (plain scores: tau = 1, no noise)
    p.cs = (float)(kLog2e / sqrt((double)s.head_dim) / tau);
    p.key0 = (uint32_t)seed;
    p.key1 = (uint32_t)(seed >> 32);
    p.noise_scale = (float)(kLog2e / tau);
    p.partial = a.partial;
    p.neg_bias = a.neg_bias;
    p.scores = a.scores;
    const T *q = static_cast<const T *>(a.q);
    const T *k = static_cast<const T *>(a.k);
    const size_t sm1 = (size_t)kSub * s.head_dim * sizeof(float);
    const size_t sm2 = sm1 + kSub * sizeof(float);
    cudaFuncSetAttribute(score_stats_simt<T, NOISE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sm1);
    cudaFuncSetAttribute(score_colmean_simt<T, NOISE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sm2);
    score_stats_simt<T, NOISE><<<sp.grid, kSimtThreads, sm1, st>>>(q, k, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_score: SIMT pass-1 launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    int rc = launch_score_merge(s, sp, a, st);
    if (rc || a.stats_only) return rc;
    score_colmean_simt<T, NOISE><<<sp.grid, kSimtThreads, sm2, st>>>(q, k, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_score: SIMT pass-2 launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

}  // namespace

int launch_score_merge(const kvc_shape &s, const ScoreSplit &sp, const ScoreArgs &a,
                       cudaStream_t st) {
    (void)s;
    const int64_t n = sp.n_units * sp.rows_pad;
    const int threads = 256;
    score_merge<<<(unsigned)((n + threads - 1) / threads), threads, 0, st>>>(
        a.partial, a.neg_bias, sp.n_units, sp.tiles_per_unit, sp.n_tiles, sp.grid, sp.max_slots,
        sp.rows, sp.rows_pad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_score: merge launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

int launch_score_simt(const kvc_shape &s, const ScoreSplit &sp, const ScoreArgs &a,
                      cudaStream_t st) {
    if (s.dtype == KVC_F32) return launch_simt_t<float, false>(s, sp, a, st);
    return launch_simt_t<__nv_bfloat16, false>(s, sp, a, st);
}

int launch_score_keyformer(const kvc_shape &s, const ScoreSplit &sp, const ScoreArgs &a,
                           uint64_t seed, double tau, cudaStream_t st) {
    if (s.dtype == KVC_F32) return launch_simt_t<float, true>(s, sp, a, st, seed, tau);
    return launch_simt_t<__nv_bfloat16, true>(s, sp, a, st, seed, tau);
}

}  // namespace kvc
