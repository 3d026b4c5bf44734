// score_tc.cu -- observation-window scores on the sm_103a tensor cores.
//
// What is computed (SnapKV scoring, blog post "ZigZagKV, KVCache 80%
// compression near-lossless", section "SnapKV"; attention as in "ThinK:
// Thinner Key Cache by Query-Driven Pruning", "Method details"): for every
// unit = (layer, KV head) with its R = G*W window query rows r = g*W + w,
//   s_rj   = q_r . k_j                               (bf16 in, fp32 accumulate)
//   x_rj   = s_rj * log2(e) / sqrt(D)                (base-2 logits)
//   c_j    = 1/R * sum_r 2^(x_rj - m_r) / l_r        over rows that see j
// with m_r, l_r the max and sum of 2^(x_rj - m_r) over the keys j <= T-W+w.
//
// The exact column mean needs each row's final normaliser before any column
// can be summed, so the contraction runs twice and the R x T matrix is never
// stored:
//   pass 1  D = Q K^T (M = 128 query rows per MMA, N = 128 keys): each
//           epilogue thread owns one TMEM lane = one query row and keeps an
//           online (max, sum) over its CTA's keys -> per-CTA partials;
//   merge   (score_simt.cu) combines the partials into nb_r = -(m_r + log2 l_r);
//   pass 2  D = K Q^T (M = 128 keys per MMA, N <= 256 query rows): each
//           epilogue thread owns one key and sums 2^(x_rj + nb_r) over the
//           query rows in registers -- the column sum needs no cross-lane
//           reduction in this orientation.
//
// Both passes are persistent: CTA c owns a contiguous run of (unit, key
// tile) pairs, keeps the unit's Q block resident in shared memory and streams
// K tiles with TMA through an mbarrier ring.  Warp roles: warp 0 TMA
// producer, warp 1 MMA issuer (and TMEM owner), warps 2-5 epilogue.  Every
// wait is bounded (kvc_internal.cuh).
#include "kvc_internal.cuh"

#include <cstdio>
#include <cstring>
#include <cudaTypedefs.h>

namespace kvc {

namespace {

constexpr int kThreads = 192;     // 6 warps
constexpr int kEpiThreads = 128;  // warps 2..5
constexpr uint32_t kTmemCols = 512;
constexpr int kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 64 bf16

struct TcParams {
    int64_t n_tiles;
    int64_t tiles_per_unit;
    int grid;
    int max_slots;
    int T, P, W;
    int rows;       // G*W
    int rows_pad;   // multiple of 128
    int n_pad;      // rows rounded up to 16 (pass-2 MMA N extent)
    int stages;
    float cs;       // log2(e) / sqrt(D)
    float2 *partial;
    const float *neg_bias_in;
    float *scores;
    uint32_t *status;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Shared-memory carve-up common to both passes.
struct Smem {
    uint8_t *q;        // [KH][rows_pad][128 B], 128-byte swizzled (TMA)
    uint8_t *k;        // [stages][KH][128 keys][128 B]
    float *nb;         // [rows_pad] (pass 2)
    int *wr;           // [rows_pad] window position of each row (pass 2)
    uint64_t *full, *empty, *q_full, *q_empty, *t_full, *t_empty, *drain;
    uint32_t *tmem_base;
    volatile int *abort_flag;
};

template <int KH>
__device__ __forceinline__ Smem carve(uint8_t *raw, const TcParams &p) {
    Smem s;
    uint8_t *b = align1024(raw);
    s.q = b;
    b += (size_t)KH * p.rows_pad * 128;
    s.k = b;
    b += (size_t)p.stages * KH * kBoxBytes;
    s.nb = reinterpret_cast<float *>(b);
    b += (size_t)p.rows_pad * sizeof(float);
    s.wr = reinterpret_cast<int *>(b);
    b += (size_t)p.rows_pad * sizeof(int);
    uint64_t *bars = reinterpret_cast<uint64_t *>(b);
    s.full = bars;
    s.empty = bars + p.stages;
    s.q_full = bars + 2 * p.stages;
    s.q_empty = s.q_full + 1;
    s.t_full = s.q_empty + 1;   // 4
    s.t_empty = s.t_full + 4;   // 4
    s.drain = s.t_empty + 4;
    s.tmem_base = reinterpret_cast<uint32_t *>(s.drain + 1);
    s.abort_flag = reinterpret_cast<volatile int *>(s.tmem_base + 1);
    return s;
}

template <int KH>
size_t smem_bytes(int rows_pad, int stages) {
    return 1024 + (size_t)KH * rows_pad * 128 + (size_t)stages * KH * kBoxBytes +
           (size_t)rows_pad * 8 + (size_t)(2 * stages + 11) * 8 + 16;
}

// Barrier set-up, TMEM allocation; returns the TMEM base column address.
__device__ __forceinline__ uint32_t setup(const Smem &s, const TcParams &p) {
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        mbar_init(s.q_full, 1);
        mbar_init(s.q_empty, 1);
        for (int i = 0; i < 4; ++i) {
            mbar_init(&s.t_full[i], 1);
            mbar_init(&s.t_empty[i], 4);  // one arrive per epilogue warp
        }
        mbar_init(s.drain, 1);
        *s.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(s.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return *s.tmem_base;
}

// TMA producer (one thread): the unit's Q block whenever the unit changes,
// then one K tile per stage.  Returns after draining its own copies.
template <int KH>
__device__ void producer(const Smem &s, const TcParams &p, const CUtensorMap *tq,
                         const CUtensorMap *tk, int64_t t0, int64_t t1) {
    int stage = 0;
    uint32_t phase = 0;
    uint32_t q_loads = 0;
    int64_t issued = 0;
    for (int64_t t = t0; t < t1; ++t) {
        const int u = (int)(t / p.tiles_per_unit);
        const int jt = (int)(t % p.tiles_per_unit);
        if (t == t0 || jt == 0) {
            if (q_loads > 0 && !mbar_wait(s.q_empty, (q_loads - 1) & 1, s.abort_flag, p.status))
                break;
            mbar_arrive_expect_tx(s.q_full, (uint32_t)(KH * p.rows_pad * 128));
            for (int kh = 0; kh < KH; ++kh)
                for (int rb = 0; rb < p.rows_pad / 128; ++rb)
                    tma_load_3d(tq, s.q_full, s.q + ((size_t)kh * p.rows_pad + rb * 128) * 128,
                                kh * 64, rb * 128, u);
            ++q_loads;
        }
        if (!mbar_wait(&s.empty[stage], phase ^ 1, s.abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&s.full[stage], (uint32_t)(KH * kBoxBytes));
        for (int kh = 0; kh < KH; ++kh)
            tma_load_3d(tk, &s.full[stage], s.k + ((size_t)stage * KH + kh) * kBoxBytes, kh * 64,
                        jt * kTileKeys, u);
        ++issued;
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1;
        }
    }
    // Unwind: every copy this thread started must land before the CTA exits.
    // In the normal case the consumer already saw them all complete.
    if (*s.abort_flag) {
        for (int64_t i = issued > p.stages ? issued - p.stages : 0; i < issued; ++i)
            mbar_drain(&s.full[i % p.stages], (uint32_t)((i / p.stages) & 1));
        if (q_loads > 0) mbar_drain(s.q_full, (q_loads - 1) & 1);
    }
}

__device__ __forceinline__ void mma_drain(const Smem &s) {
    tc_commit(s.drain);
    mbar_drain(s.drain, 0);
}

// --------------------------------------------------------------- pass 1
template <int KH>
__global__ void __launch_bounds__(kThreads, 1)
    score_stats_tc(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve<KH>(smem_raw, p);
    const uint32_t tmem = setup(s, p);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c = blockIdx.x;
    const int64_t t0 = split_begin(p.n_tiles, p.grid, c), t1 = split_begin(p.n_tiles, p.grid, c + 1);
    const int nrb = p.rows_pad / 128;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            producer<KH>(s, p, &tq, &tk, t0, t1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, kTileKeys);
            int stage = 0;
            uint32_t phase = 0, q_loads = 0;
            uint32_t job = 0;
            bool ok = true;
            for (int64_t t = t0; t < t1 && ok; ++t) {
                const int jt = (int)(t % p.tiles_per_unit);
                const bool last = (t == t1 - 1) || (jt == p.tiles_per_unit - 1);
                if (t == t0 || jt == 0) {
                    if (!mbar_wait(s.q_full, q_loads & 1, s.abort_flag, p.status)) break;
                    ++q_loads;
                }
                if (!mbar_wait(&s.full[stage], phase, s.abort_flag, p.status)) break;
                tc_fence_after();
                for (int rb = 0; rb < nrb; ++rb, ++job) {
                    const uint32_t slot = job & 3, use = job >> 2;
                    if (!mbar_wait(&s.t_empty[slot], (use & 1) ^ 1, s.abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + slot * 128;
#pragma unroll
                    for (int ks = 0; ks < KH * 4; ++ks) {
                        const int kh = ks >> 2, off = (ks & 3) * 32;
                        const uint64_t a = sw128_kmajor_desc(
                            smem_u32(s.q + ((size_t)kh * p.rows_pad + rb * 128) * 128) + off);
                        const uint64_t b = sw128_kmajor_desc(
                            smem_u32(s.k + ((size_t)stage * KH + kh) * kBoxBytes) + off);
                        tc_mma_bf16(d, a, b, idesc, ks > 0);
                    }
                    tc_commit(&s.t_full[slot]);
                }
                if (!ok) break;
                tc_commit(&s.empty[stage]);
                if (last) tc_commit(s.q_empty);
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            mma_drain(s);
        }
    } else {
        // Epilogue: TMEM lane quarter is fixed by warp id % 4.
        const int quarter = warp & 3;
        const int row_in_blk = quarter * 32 + lane;
        float m_run[4], l_run[4];
        uint32_t job = 0;
        bool ok = true;
        for (int64_t t = t0; t < t1 && ok; ++t) {
            const int u = (int)(t / p.tiles_per_unit);
            const int jt = (int)(t % p.tiles_per_unit);
            const int j0 = jt * kTileKeys;
            const bool last = (t == t1 - 1) || (jt == p.tiles_per_unit - 1);
            if (t == t0 || jt == 0) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    m_run[i] = -INFINITY;
                    l_run[i] = 0.f;
                }
            }
            const bool masked = j0 + kTileKeys - 1 > p.P;
#pragma unroll
            for (int rb = 0; rb < 4; ++rb) {
                if (rb >= nrb) break;
                const uint32_t slot = job & 3, use = job >> 2;
                ++job;
                if (!mbar_wait(&s.t_full[slot], use & 1, s.abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + slot * 128;
                float v[128];
                tmem_ld32(taddr + 0, *reinterpret_cast<float(*)[32]>(&v[0]));
                tmem_ld32(taddr + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
                tmem_ld32(taddr + 64, *reinterpret_cast<float(*)[32]>(&v[64]));
                tmem_ld32(taddr + 96, *reinterpret_cast<float(*)[32]>(&v[96]));
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.t_empty[slot]);

                const int r = rb * 128 + row_in_blk;
                float mx = -INFINITY, sum = 0.f, mnew;
                if (!masked) {
#pragma unroll
                    for (int i = 0; i < 128; ++i) mx = fmaxf(mx, v[i]);
                    mnew = fmaxf(m_run[rb], mx * p.cs);
#pragma unroll
                    for (int i = 0; i < 128; ++i) sum += ex2(fmaf(v[i], p.cs, -mnew));
                } else {
                    // Largest column of this tile that row r may see.
                    const int lim = p.P + (r % p.W) - j0;
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (i <= lim) mx = fmaxf(mx, v[i]);
                    mnew = fmaxf(m_run[rb], mx * p.cs);
                    if (mx > -INFINITY) {
#pragma unroll
                        for (int i = 0; i < 128; ++i)
                            if (i <= lim) sum += ex2(fmaf(v[i], p.cs, -mnew));
                    }
                }
                if (mx > -INFINITY) {
                    l_run[rb] = l_run[rb] * ex2(m_run[rb] - mnew) + sum;
                    m_run[rb] = mnew;
                }
            }
            if (!ok) break;
            if (last) {
                const int64_t slot_u = c - split_cta_of(p.n_tiles, p.grid, (int64_t)u * p.tiles_per_unit);
                float2 *dst = p.partial + ((int64_t)u * p.max_slots + slot_u) * p.rows_pad;
#pragma unroll
                for (int rb = 0; rb < 4; ++rb) {
                    const int r = rb * 128 + row_in_blk;
                    if (rb < nrb && r < p.rows) dst[r] = make_float2(m_run[rb], l_run[rb]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// --------------------------------------------------------------- pass 2
template <int KH>
__global__ void __launch_bounds__(kThreads, 1)
    score_colmean_tc(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve<KH>(smem_raw, p);
    const uint32_t tmem = setup(s, p);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c = blockIdx.x;
    const int64_t t0 = split_begin(p.n_tiles, p.grid, c), t1 = split_begin(p.n_tiles, p.grid, c + 1);
    const int nch = (p.n_pad + 255) / 256;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            producer<KH>(s, p, &tq, &tk, t0, t1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, q_loads = 0;
            uint32_t job = 0;
            bool ok = true;
            for (int64_t t = t0; t < t1 && ok; ++t) {
                const int jt = (int)(t % p.tiles_per_unit);
                const bool last = (t == t1 - 1) || (jt == p.tiles_per_unit - 1);
                if (t == t0 || jt == 0) {
                    if (!mbar_wait(s.q_full, q_loads & 1, s.abort_flag, p.status)) break;
                    ++q_loads;
                }
                if (!mbar_wait(&s.full[stage], phase, s.abort_flag, p.status)) break;
                tc_fence_after();
                for (int nc = 0; nc < nch; ++nc, ++job) {
                    const uint32_t slot = job & 1, use = job >> 1;
                    if (!mbar_wait(&s.t_empty[slot], (use & 1) ^ 1, s.abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int n = min(256, p.n_pad - nc * 256);
                    const uint32_t idesc = idesc_bf16_f32(128, n);
                    const uint32_t d = tmem + slot * 256;
#pragma unroll
                    for (int ks = 0; ks < KH * 4; ++ks) {
                        const int kh = ks >> 2, off = (ks & 3) * 32;
                        const uint64_t a = sw128_kmajor_desc(
                            smem_u32(s.k + ((size_t)stage * KH + kh) * kBoxBytes) + off);
                        const uint64_t b = sw128_kmajor_desc(
                            smem_u32(s.q + ((size_t)kh * p.rows_pad + nc * 256) * 128) + off);
                        tc_mma_bf16(d, a, b, idesc, ks > 0);
                    }
                    tc_commit(&s.t_full[slot]);
                }
                if (!ok) break;
                tc_commit(&s.empty[stage]);
                if (last) tc_commit(s.q_empty);
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            mma_drain(s);
        }
    } else {
        const int quarter = warp & 3;
        const int etid = threadIdx.x - 64;   // 0..127 over the epilogue warps
        const int key_in_tile = quarter * 32 + lane;
        const float rows_f = (float)p.rows;
        uint32_t job = 0;
        bool ok = true;
        float acc = 0.f;
        for (int64_t t = t0; t < t1 && ok; ++t) {
            const int u = (int)(t / p.tiles_per_unit);
            const int jt = (int)(t % p.tiles_per_unit);
            const int j0 = jt * kTileKeys;
            if (t == t0 || jt == 0) {
                named_bar_sync(1, kEpiThreads);
                for (int r = etid; r < p.rows_pad; r += kEpiThreads) {
                    s.nb[r] = p.neg_bias_in[(int64_t)u * p.rows_pad + r];
                    s.wr[r] = r < p.rows ? r % p.W : p.W;
                }
                named_bar_sync(1, kEpiThreads);
            }
            const int j = j0 + key_in_tile;
            const int dj = j - p.P;   // row r sees key j iff wr[r] >= dj
            const bool masked = j0 + kTileKeys - 1 > p.P;
            for (int nc = 0; nc < nch; ++nc) {
                const uint32_t slot = job & 1, use = job >> 1;
                ++job;
                if (!mbar_wait(&s.t_full[slot], use & 1, s.abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int n = min(256, p.n_pad - nc * 256);
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + slot * 256;
                const float *nb = s.nb + nc * 256;
                const int *wr = s.wr + nc * 256;
                for (int cg = 0; cg < n; cg += 32) {
                    float v[32];
                    const int cnt = min(32, n - cg);
                    if (cnt == 32) {
                        tmem_ld32(taddr + cg, v);
                    } else {
                        tmem_ld16(taddr + cg, *reinterpret_cast<float(*)[16]>(&v[0]));
                    }
                    tmem_ld_wait();
                    if (!masked) {
                        if (cnt == 32) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) acc += ex2(fmaf(v[i], p.cs, nb[cg + i]));
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) acc += ex2(fmaf(v[i], p.cs, nb[cg + i]));
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            if (i < cnt) {
                                const float e = ex2(fmaf(v[i], p.cs, nb[cg + i]));
                                acc += (wr[cg + i] >= dj) ? e : 0.f;
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.t_empty[slot]);
            }
            if (!ok) break;
            if (j < p.T) p.scores[(int64_t)u * p.T + j] = acc / rows_f;
            acc = 0.f;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// --------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 3-D bf16 view [outer][mid][inner] with a (64, 128, 1) box, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t mid, uint64_t outer) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {inner, mid, outer};
    cuuint64_t strides[2] = {inner * 2, inner * mid * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int KH>
int launch_kh(const kvc_shape &s, const ScoreSplit &sp, const ScoreArgs &a, cudaStream_t st) {
    const int G = s.n_q_heads / s.n_kv_heads;
    CUtensorMap tq, tk;
    if (!make_map(&tq, a.q, (uint64_t)s.head_dim, (uint64_t)G * s.window, (uint64_t)sp.n_units) ||
        !make_map(&tk, a.k, (uint64_t)s.head_dim, (uint64_t)s.seq_len, (uint64_t)sp.n_units)) {
        set_error("kvc_score: cuTensorMapEncodeTiled failed (alignment or driver)");
        return KVC_ERR_CUDA;
    }
    TcParams p;
    p.n_tiles = sp.n_tiles;
    p.tiles_per_unit = sp.tiles_per_unit;
    p.grid = sp.grid;
    p.max_slots = sp.max_slots;
    p.T = s.seq_len;
    p.W = s.window;
    p.P = s.seq_len - s.window;
    p.rows = sp.rows;
    p.rows_pad = sp.rows_pad;
    p.n_pad = (sp.rows + 15) / 16 * 16;
    p.cs = (float)(kLog2e / sqrt((double)s.head_dim));
    p.partial = a.partial;
    p.neg_bias_in = a.neg_bias;
    p.scores = a.scores;
    p.status = a.status;
    // Deepest K ring that fits next to the resident Q block.
    int stages = 4;
    while (stages > 2 && smem_bytes<KH>(sp.rows_pad, stages) > 232448) --stages;
    p.stages = stages;
    const size_t smem = smem_bytes<KH>(sp.rows_pad, stages);
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(score_stats_tc<KH>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
        cudaFuncSetAttribute(score_colmean_tc<KH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             232448);
        attr_set = true;
    }
    score_stats_tc<KH><<<sp.grid, kThreads, smem, st>>>(tq, tk, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_score: pass-1 launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    int rc = launch_score_merge(s, sp, a, st);
    if (rc) return rc;
    score_colmean_tc<KH><<<sp.grid, kThreads, smem, st>>>(tq, tk, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_score: pass-2 launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

}  // namespace

int launch_score_tc(const kvc_shape &s, const ScoreSplit &sp, const ScoreArgs &a, int num_sms,
                    cudaStream_t st) {
    (void)num_sms;
    if (s.head_dim == 128) return launch_kh<2>(s, sp, a, st);
    if (s.head_dim == 64) return launch_kh<1>(s, sp, a, st);
    set_error("kvc_score: tensor-core path needs head_dim 64 or 128");
    return KVC_ERR_UNSUPPORTED;
}

}  // namespace kvc
