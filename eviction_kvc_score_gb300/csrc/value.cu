// value.cu -- ThinK value-channel scores (THINKV).
//
// "ThinK: Thinner Key Cache by Query-Driven Pruning", appendix "Value cache
// pruning strategy": channel j of a head's value cache scores the norm of
// column j of the window queries' attention output,
//   Score_v[j] = || softmax(Q_obs K^T / sqrt(D)) V[:, j] ||,
// and the top floor((1-lambda) D) channels are kept.  Here, per unit = (layer,
// KV head) with its R = G*W window rows r = g*W + w (row r at position P + w
// sees keys j <= P + w):
//   o_r[d]     = sum_j 2^(x_rj + nb_r) v_j[d],   x_rj = q_r . k_j log2(e)/sqrt(D)
//   score_v[d] = sum_r o_r[d]^2                  (the squared norm: same order)
// with nb_r = -(m_r + log2 l_r) the row's softmax normaliser from the score
// pass's first half (pass 1 + merge), so every probability is exact when it
// is formed and the output needs no rescaling.
//
// This file holds the CUDA-core kernel (every dtype and head_dim), the
// deterministic merge of per-part sums, and the dispatch; the tensor-core
// kernel for bf16 / head_dim 128 lives in value_tc.cu.
#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int kVThreads = 128;
constexpr int kVRows = 16;   // window rows per block
constexpr int kVKeys = 32;   // keys per shared-memory tile
constexpr int kVParts = 16;  // blocks (partial sums) per unit at most

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

struct VParams {
    int T, P, W, D, rows, rows_pad, chunks;
    int parts;                // blocks per unit: block b takes chunks b, b + parts, ...
    float cs;                 // log2(e) / sqrt(D)
    const float *neg_bias;    // [units][rows_pad]
    float *partial;           // [units][parts][D]
};

// Block (part, unit) handles the unit's 16-row chunks part, part + parts, ...
// in that order; for each chunk the keys and values stream through shared
// memory 32 at a time, thread (key j, row group) forms 4 logits, then thread d
// accumulates o_r[d] for the 16 rows (and d + 128 when D > 128) and adds
// o_r[d]^2 to its running sum.  At the end each thread writes its sum: one
// partial per (unit, part), at most kVParts per unit.
template <typename T>
__global__ void __launch_bounds__(kVThreads)
    value_out_simt(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                   VParams p) {
    extern __shared__ float sm[];
    const int D = p.D, DK = D + 1;                   // key rows padded: no bank conflicts
    float *qs = sm;                                  // [16][D]
    float *ks = qs + kVRows * D;                     // [32][D+1]
    float *vs = ks + kVKeys * DK;                    // [32][D]
    float *ps = vs + kVKeys * D;                     // [16][32]
    float *nb = ps + kVRows * kVKeys;                // [16]
    const int64_t u = blockIdx.y;
    const int tid = threadIdx.x;
    float sq[2] = {0.f, 0.f};
    for (int chunk = blockIdx.x; chunk < p.chunks; chunk += p.parts) {
        const int r0 = chunk * kVRows;
        __syncthreads();   // the previous chunk's shared memory is no longer read
        for (int e = tid; e < kVRows * D; e += kVThreads) {
            const int r = r0 + e / D;
            qs[e] = r < p.rows ? to_f(q[(u * p.rows + r) * (int64_t)D + e % D]) : 0.f;
        }
        if (tid < kVRows) {
            const int r = r0 + tid;
            nb[tid] = r < p.rows ? p.neg_bias[u * p.rows_pad + r] : -INFINITY;
        }
        // the last window position a row of this chunk sees
        const int r_last = min(r0 + kVRows, p.rows) - 1;
        int w_max = 0;
        for (int r = r0; r <= r_last; ++r) w_max = max(w_max, r % p.W);
        const int j_end = min(p.T, p.P + w_max + 1);
        const int jk = tid & 31, rg = tid >> 5;          // logits: key jk, rows 4 rg .. 4 rg + 3
        float acc[kVRows][2];
#pragma unroll
        for (int r = 0; r < kVRows; ++r) acc[r][0] = acc[r][1] = 0.f;
        const T *ku = k + u * (int64_t)p.T * D;
        const T *vu = v + u * (int64_t)p.T * D;
        for (int j0 = 0; j0 < j_end; j0 += kVKeys) {
            __syncthreads();
            for (int e = tid; e < kVKeys * D; e += kVThreads) {
                const int jj = j0 + e / D, d = e % D;
                const bool in = jj < p.T;
                ks[(e / D) * DK + d] = in ? to_f(ku[(int64_t)jj * D + d]) : 0.f;
                vs[e] = in ? to_f(vu[(int64_t)jj * D + d]) : 0.f;
            }
            __syncthreads();
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
            for (int d = 0; d < D; ++d) {
                const float kd = ks[jk * DK + d];
#pragma unroll
                for (int i = 0; i < 4; ++i) s4[i] = fmaf(qs[(rg * 4 + i) * D + d], kd, s4[i]);
            }
            const int j = j0 + jk;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int rl = rg * 4 + i, r = r0 + rl;
                const bool vis = r < p.rows && j < p.T && j <= p.P + r % p.W;
                ps[rl * kVKeys + jk] = vis ? ex2(fmaf(s4[i], p.cs, nb[rl])) : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int d = tid + h * kVThreads;
                if (d < D) {
#pragma unroll 4
                    for (int jj = 0; jj < kVKeys; ++jj) {
                        const float vd = vs[jj * D + d];
#pragma unroll
                        for (int r = 0; r < kVRows; ++r) acc[r][h] = fmaf(ps[r * kVKeys + jj], vd, acc[r][h]);
                    }
                }
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int r = 0; r < kVRows; ++r) sq[h] = fmaf(acc[r][h], acc[r][h], sq[h]);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int d = tid + h * kVThreads;
        if (d < D) p.partial[(u * p.parts + blockIdx.x) * (int64_t)D + d] = sq[h];
    }
}

// score_v[u][d] = sum over the unit's first `parts` parts (of `stride` per
// unit), in part order (deterministic).
__global__ void value_merge(const float *__restrict__ partial, int parts, int stride, int D,
                            int64_t units, float *__restrict__ score_v) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= units * D) return;
    const int64_t u = i / D;
    const int d = (int)(i % D);
    const float *pp = partial + u * (int64_t)stride * D + d;
    float s = 0.f;
    for (int c = 0; c < parts; ++c) s += pp[(int64_t)c * D];
    score_v[i] = s;
}

template <typename T>
int launch_simt_t(const kvc_shape &s, const ScoreSplit &sp, const void *q, const void *k,
                  const void *v, const float *neg_bias, float *partial, cudaStream_t st,
                  int *parts_out) {
    VParams p;
    p.T = s.seq_len;
    p.P = s.seq_len - s.window;
    p.W = s.window;
    p.D = s.head_dim;
    p.rows = sp.rows;
    p.rows_pad = sp.rows_pad;
    p.chunks = (sp.rows + kVRows - 1) / kVRows;
    p.parts = p.chunks < kVParts ? p.chunks : kVParts;
    p.cs = (float)(kLog2e / sqrt((double)s.head_dim));
    p.neg_bias = neg_bias;
    p.partial = partial;
    const size_t smem = sizeof(float) * ((size_t)kVRows * p.D + (size_t)kVKeys * (p.D + 1) +
                                         (size_t)kVKeys * p.D + kVRows * kVKeys + kVRows);
    cudaFuncSetAttribute(value_out_simt<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    value_out_simt<T><<<dim3((unsigned)p.parts, (unsigned)sp.n_units), kVThreads, smem, st>>>(
        static_cast<const T *>(q), static_cast<const T *>(k), static_cast<const T *>(v), p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_channel_prune_value: value-output launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    *parts_out = p.parts;
    return KVC_OK;
}

}  // namespace

int64_t value_partial_floats(const kvc_shape &s) {
    const int64_t parts = kVParts > kValueTcParts ? kVParts : kValueTcParts;
    return (int64_t)s.n_layers * s.n_kv_heads * parts * s.head_dim;
}

int launch_value_scores(const kvc_shape &s, const ScoreSplit &sp, const void *q, const void *k,
                        const void *v, const float *neg_bias, float *partial, float *score_v,
                        bool tc, uint32_t *status, cudaStream_t st) {
    int parts = 0, rc;
    if (tc)
        rc = launch_value_tc(s, sp, q, k, v, neg_bias, partial, status, st, &parts);
    else if (s.dtype == KVC_F32)
        rc = launch_simt_t<float>(s, sp, q, k, v, neg_bias, partial, st, &parts);
    else
        rc = launch_simt_t<__nv_bfloat16>(s, sp, q, k, v, neg_bias, partial, st, &parts);
    if (rc) return rc;
    const int64_t n = sp.n_units * s.head_dim;
    const int stride = tc ? kValueTcParts : parts;
    value_merge<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(partial, parts, stride, s.head_dim,
                                                              sp.n_units, score_v);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_channel_prune_value: merge launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

}  // namespace kvc
