// pool.cu -- optional SnapKV 1D pooling of the prefix scores before top-K.
//
// Blog post "ZigZagKV, KVCache 80% compression near-lossless", section
// "SnapKV": after the window-mean scores are formed, each head's scores are
// pooled in 1D so that the neighbours of an important token are kept with it
// (the post likens it to a Gaussian blur).  The post gives neither the kernel
// size nor its type; this library takes an odd kernel k and either averages
// the in-range prefix neighbours j-k/2 .. j+k/2 (dividing by how many of them
// lie inside the prefix) or takes their maximum.  Window positions are
// copied unchanged.
//
// Work split: one block per (1024-position tile, head); the tile and its
// k-1 halo are staged in shared memory with coalesced loads.  Each thread
// produces four outputs 256 apart, summing their taps left to right in fp32
// in one loop so that the four dependency chains overlap.
#include <algorithm>

#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int kPoolTile = 1024;
constexpr int kPoolThreads = 256;
constexpr int kPoolPer = kPoolTile / kPoolThreads;   // outputs per thread
constexpr int kPoolMaxKernel = 255;

__global__ void __launch_bounds__(kPoolThreads)
    pool_kernel(const float *__restrict__ scores, int64_t n_heads, int T, int P, int kernel,
                int mode, float *__restrict__ pooled) {
    __shared__ float tile[kPoolTile + kPoolMaxKernel];
    const int j0 = blockIdx.x * kPoolTile;
    const int half = kernel / 2;
    for (int64_t head = blockIdx.y; head < n_heads; head += gridDim.y) {
        const float *c = scores + head * T;
        float *o = pooled + head * T;
        __syncthreads();   // the previous head's tile is no longer read
        // tile[i] holds position j0 - half + i (0 outside [0, T): never used
        // by an output, which reads only positions inside the prefix)
        for (int i = threadIdx.x; i < kPoolTile + kernel - 1; i += kPoolThreads) {
            const int t = j0 - half + i;
            tile[i] = (t >= 0 && t < T) ? c[t] : 0.f;
        }
        __syncthreads();
        const int jb = j0 + threadIdx.x;   // this thread's outputs: jb + u * kPoolThreads
        const int jl = jb + (kPoolPer - 1) * kPoolThreads;
        if (jb - half >= 0 && jl + half < P) {
            // all four outputs see a full kernel inside the prefix
            float acc[kPoolPer];
#pragma unroll
            for (int u = 0; u < kPoolPer; ++u) acc[u] = tile[threadIdx.x + u * kPoolThreads];
#pragma unroll 4
            for (int t = 1; t < kernel; ++t) {
#pragma unroll
                for (int u = 0; u < kPoolPer; ++u) {
                    const float x = tile[threadIdx.x + u * kPoolThreads + t];
                    acc[u] = mode == 0 ? acc[u] + x : fmaxf(acc[u], x);
                }
            }
#pragma unroll
            for (int u = 0; u < kPoolPer; ++u)
                o[jb + u * kPoolThreads] = mode == 0 ? acc[u] / (float)kernel : acc[u];
            continue;
        }
        for (int u = 0; u < kPoolPer; ++u) {
            const int j = jb + u * kPoolThreads;
            if (j >= T) break;
            if (j >= P) {
                o[j] = tile[j - j0 + half];
                continue;
            }
            const int lo = max(0, j - half), hi = min(P - 1, j + half);
            float acc = tile[lo - j0 + half];
            for (int t = lo + 1; t <= hi; ++t) {
                const float x = tile[t - j0 + half];
                acc = mode == 0 ? acc + x : fmaxf(acc, x);
            }
            o[j] = mode == 0 ? acc / (float)(hi - lo + 1) : acc;
        }
    }
}

}  // namespace

int launch_pool(const kvc_shape &s, const float *scores, int32_t kernel, int32_t mode, float *pooled,
                cudaStream_t st) {
    if (kernel > kPoolMaxKernel) {
        set_error("kvc_pool_scores: kernel above %d is not supported", kPoolMaxKernel);
        return KVC_ERR_UNSUPPORTED;
    }
    const int64_t n_heads = (int64_t)s.n_layers * s.n_kv_heads;
    dim3 grid((s.seq_len + kPoolTile - 1) / kPoolTile, (unsigned)std::min<int64_t>(n_heads, 65535));
    pool_kernel<<<grid, kPoolThreads, 0, st>>>(scores, n_heads, s.seq_len, s.seq_len - s.window,
                                               kernel, mode, pooled);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_pool_scores: launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

}  // namespace kvc
