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
//   pass 2  D = K Q^T (M = 128 keys per MMA, N <= 256 query rows) plus one
//           extra K-step that adds nb_r / (log2(e)/sqrt(D)) to every column r
//           (ones against the row biases split into three bf16 terms): each
//           epilogue thread owns one key and sums 2^(x'_rj) over the query
//           rows in registers -- no cross-lane reduction in this orientation,
//           and no per-logit bias load.
//
// Both passes are persistent: CTA c owns a contiguous run of (unit, key
// tile) pairs, keeps the unit's Q block resident in shared memory and streams
// K tiles with TMA through an mbarrier ring.  Warp roles: warp 0 TMA
// producer, warp 1 MMA issuer (and TMEM owner), warps 2-9 epilogue in two
// warpgroups.  Pass 1 splits TMEM into four 128-column accumulator slots
// (one 128 x 128 job each; the warpgroups take alternate jobs); pass 2 into
// two 256-column slots (one 128 x 256 job each: with both operands in shared
// memory the wider MMA reads fewer operand bytes per flop), each job's
// columns split between the two warpgroups so that a slot is free again
// after two TMEM loads per warp.  A job is read from TMEM in 64-column
// pieces; each thread keeps independent sum chains on packed fp32 pairs, and
// the epilogue has one copy of its inner loop (the window's causal mask is
// applied by setting invisible logits to -inf first) so that it fits the
// instruction cache.  Measured on this GPU, shared-memory loads in the
// epilogue compete with the MMAs' shared-memory operand reads (an exp loop
// with them runs at half speed beside the MMA stream, without them at full
// speed), which is why pass 2 takes the row biases through the MMA; and
// every instruction per logit counts, which is why pass 1 keeps a running
// reference that is raised only when a piece would overflow instead of
// taking every piece's maximum.
// Every wait is bounded (kvc_internal.cuh); there are no named barriers.
#include "kvc_internal.cuh"

#include <cstdio>
#include <cstring>
#include <cudaTypedefs.h>

namespace kvc {

namespace {

constexpr int kThreads = 320;     // 10 warps: producer, MMA, 2 x 4 epilogue
constexpr int kEpi = 256;         // epilogue threads
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
    uint8_t *aug_k;    // [128 keys][32 B] pass-2 extra K-step operand: ones
    uint8_t *aug_q;    // [rows_pad][32 B] pass-2 extra K-step operand: row biases
    float *red;        // [2][128] pass-2 partial column sums handed WG1 -> WG0
    uint64_t *full, *empty, *q_full, *q_empty, *t_full, *t_empty, *c_full, *c_empty;
    uint64_t *aug_full, *aug_empty, *drain;
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
    s.aug_k = b;
    b += 128 * 32;
    s.aug_q = b;
    b += (size_t)p.rows_pad * 32;
    s.red = reinterpret_cast<float *>(b);
    b += 2 * 128 * sizeof(float);
    uint64_t *bars = reinterpret_cast<uint64_t *>(b);
    s.full = bars;
    s.empty = bars + p.stages;
    s.q_full = bars + 2 * p.stages;
    s.q_empty = s.q_full + 1;
    s.t_full = s.q_empty + 1;   // 4
    s.t_empty = s.t_full + 4;   // 4
    s.c_full = s.t_empty + 4;   // 2
    s.c_empty = s.c_full + 2;   // 2
    s.aug_full = s.c_empty + 2;
    s.aug_empty = s.aug_full + 1;
    s.drain = s.aug_empty + 1;
    s.tmem_base = reinterpret_cast<uint32_t *>(s.drain + 1);
    s.abort_flag = reinterpret_cast<volatile int *>(s.tmem_base + 1);
    return s;
}

template <int KH>
size_t smem_bytes(int rows_pad, int stages) {
    return 1024 + (size_t)KH * rows_pad * 128 + (size_t)stages * KH * kBoxBytes + 128 * 32 +
           (size_t)rows_pad * 32 + 2 * 128 * 4 + (size_t)(2 * stages + 17) * 8 + 16;
}

// Barrier set-up, TMEM allocation; returns the TMEM base column address.
__device__ __forceinline__ uint32_t setup(const Smem &s, const TcParams &p, int t_empty_count) {
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
            mbar_init(&s.t_empty[i], t_empty_count);  // one arrive per warp reading the slot
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.c_full[i], 128);
            mbar_init(&s.c_empty[i], 128);
        }
        mbar_init(s.aug_full, kEpi);
        mbar_init(s.aug_empty, 1);
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

// K-major operand in the 32-byte swizzled layout: rows of 32 bytes (16
// bf16, one MMA K-step), 8-row groups 256 bytes apart (stride offset 256),
// layout code 6 in bits [61,64).
__device__ __forceinline__ uint64_t sw32_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(256 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(6) << 61;
    return d;
}

// MMA issuer (one thread).  For every K tile: njob jobs of fp32 accumulators
// into TMEM.  Pass 1 (KEYS_AS_B): 128 x 128 jobs into slot job % 4, A = Q
// row block jb, B = the K tile.  Pass 2: 128 x n jobs (n <= 256) into slot
// job % 2, A = the K tile, B = Q rows 256 jb ...
template <int KH, bool KEYS_AS_B>
__device__ void mma_issuer(const Smem &s, const TcParams &p, uint32_t tmem, int64_t t0, int64_t t1,
                           int njob) {
    int stage = 0;
    uint32_t phase = 0, q_loads = 0, job = 0;
    bool ok = true;
    for (int64_t t = t0; t < t1 && ok; ++t) {
        const int jt = (int)(t % p.tiles_per_unit);
        const bool last = (t == t1 - 1) || (jt == p.tiles_per_unit - 1);
        if (t == t0 || jt == 0) {
            if (!mbar_wait(s.q_full, q_loads & 1, s.abort_flag, p.status)) break;
            // pass 2 also needs the unit's row-bias operand
            if (!KEYS_AS_B && !mbar_wait(s.aug_full, q_loads & 1, s.abort_flag, p.status)) break;
            ++q_loads;
        }
        if (!mbar_wait(&s.full[stage], phase, s.abort_flag, p.status)) break;
        tc_fence_after();
        for (int jb = 0; jb < njob; ++jb, ++job) {
            constexpr uint32_t kSlots = KEYS_AS_B ? 4 : 2;
            constexpr int kCols = KEYS_AS_B ? 128 : 256;   // TMEM columns per slot
            const uint32_t slot = job % kSlots, use = job / kSlots;
            if (!mbar_wait(&s.t_empty[slot], (use & 1) ^ 1, s.abort_flag, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int n = KEYS_AS_B ? kTileKeys : min(kCols, p.n_pad - jb * kCols);
            const uint32_t idesc = idesc_bf16_f32(128, n);
            const uint32_t d = tmem + slot * kCols;
#pragma unroll
            for (int ks = 0; ks < KH * 4; ++ks) {
                const int kh = ks >> 2, off = (ks & 3) * 32;
                const uint32_t qa =
                    smem_u32(s.q + ((size_t)kh * p.rows_pad + jb * kCols) * 128) + off;
                const uint32_t ka = smem_u32(s.k + ((size_t)stage * KH + kh) * kBoxBytes) + off;
                const uint64_t a = sw128_kmajor_desc(KEYS_AS_B ? qa : ka);
                const uint64_t b = sw128_kmajor_desc(KEYS_AS_B ? ka : qa);
                tc_mma_bf16(d, a, b, idesc, ks > 0);
            }
            if (!KEYS_AS_B) {
                // one more K-step adds each query row's bias to its column:
                // ones (keys) x the row's bias / cs split into bf16 terms
                tc_mma_bf16(d, sw32_kmajor_desc(smem_u32(s.aug_k)),
                            sw32_kmajor_desc(smem_u32(s.aug_q + (size_t)jb * kCols * 32)), idesc, 1u);
            }
            tc_commit(&s.t_full[slot]);
        }
        if (!ok) break;
        tc_commit(&s.empty[stage]);
        if (last) tc_commit(s.q_empty);
        if (last && !KEYS_AS_B) tc_commit(s.aug_empty);
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1;
        }
    }
    mma_drain(s);
}

// Release a TMEM slot once this warp's loads from it have completed.
__device__ __forceinline__ void release_slot(uint64_t *bar, int lane) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

// 64 consecutive fp32 columns of this thread's TMEM lane -> v, completed.
__device__ __forceinline__ void load_row64(uint32_t taddr, float (&v)[2][32]) {
    tmem_ld32(taddr + 0, v[0]);
    tmem_ld32(taddr + 32, v[1]);
    tmem_ld_wait();
    reg_fence(v[0]);
    reg_fence(v[1]);
}

// Fold 64 logits (-inf = not visible) into a row's online (max, sum) in base
// 2, with eight independent max and sum chains.
__device__ __forceinline__ void row_stats64(const float (&v)[2][32], float cs, float &m_run,
                                            float &l_run) {
    float mx8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(v[0][i], v[0][i + 8]);
#pragma unroll
    for (int i = 16; i < 64; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], v[i >> 5][i & 31]);
    const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                           fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
    if (mx == -INFINITY) return;
    const float mnew = fmaxf(m_run, mx * cs);
    float s8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s8[i] = 0.f;
#pragma unroll
    for (int i = 0; i < 64; ++i) s8[i & 7] += ex2(fmaf(v[i >> 5][i & 31], cs, -mnew));
    const float sum = ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
    l_run = l_run * ex2(m_run - mnew) + sum;
    m_run = mnew;
}

// The same fold with a running reference that is raised only when needed:
// the piece's exponentials are taken against m_run, and if their sum stays
// below 2^60 (no logit more than ~60 above m_run, so nothing overflowed) it is
// added to l_run as it is; otherwise the piece is redone against its exact
// maximum.  Either way l_run * 2^m_run is the sum of 2^(x*cs) over the keys
// seen, which is all the merge needs; skipping the per-piece maximum removes
// one instruction per logit.  The logit arithmetic runs on packed fp32 pairs.
__device__ __forceinline__ void row_stats64_lazy(const float (&v)[2][32], float cs, float &m_run,
                                                 float &l_run) {
    if (m_run == -INFINITY) {
        row_stats64(v, cs, m_run, l_run);
        return;
    }
    unsigned long long s4[4] = {0ull, 0ull, 0ull, 0ull};
    const unsigned long long cs2 = f2_pack(cs, cs), nm2 = f2_pack(-m_run, -m_run);
#pragma unroll
    for (int i = 0; i < 64; i += 2) {
        const unsigned long long y =
            f2_fma(f2_pack(v[i >> 5][i & 31], v[i >> 5][(i & 31) + 1]), cs2, nm2);
        float y0, y1;
        f2_unpack(y, y0, y1);
        s4[(i >> 1) & 3] = f2_add(s4[(i >> 1) & 3], f2_pack(ex2(y0), ex2(y1)));
    }
    float s8[8];
    f2_unpack(s4[0], s8[0], s8[1]);
    f2_unpack(s4[1], s8[2], s8[3]);
    f2_unpack(s4[2], s8[4], s8[5]);
    f2_unpack(s4[3], s8[6], s8[7]);
    const float sum = ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
    if (sum < 0x1p60f) {
        l_run += sum;
        return;
    }
    row_stats64(v, cs, m_run, l_run);
}

// Add 2^(x * cs) for 64 query-row columns into eight partial sums; the
// accumulators already carry each row's bias nb_r / cs (packed fp32 pairs for
// the scaling and the accumulation).
__device__ __forceinline__ void col_sums64(const float (&v)[2][32], float cs, float (&a8)[8]) {
    unsigned long long a4[4] = {0ull, 0ull, 0ull, 0ull};
    const unsigned long long cs2 = f2_pack(cs, cs);
#pragma unroll
    for (int i = 0; i < 64; i += 2) {
        const unsigned long long y = f2_mul(f2_pack(v[i >> 5][i & 31], v[i >> 5][(i & 31) + 1]), cs2);
        float y0, y1;
        f2_unpack(y, y0, y1);
        a4[(i >> 1) & 3] = f2_add(a4[(i >> 1) & 3], f2_pack(ex2(y0), ex2(y1)));
    }
    float t[8];
    f2_unpack(a4[0], t[0], t[1]);
    f2_unpack(a4[1], t[2], t[3]);
    f2_unpack(a4[2], t[4], t[5]);
    f2_unpack(a4[3], t[6], t[7]);
#pragma unroll
    for (int i = 0; i < 8; ++i) a8[i] += t[i];
}

// Causal mask inside the window for pass 2: row r = g*W + w sees the key iff
// w >= dj.  w advances with the column and wraps at W; it carries over
// between consecutive chunks.
__device__ __forceinline__ void mask_cols(float (&v)[32], int &w, int dj, int W) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        if (w < dj) v[i] = -INFINITY;
        w = (w + 1 == W) ? 0 : w + 1;
    }
}

// --------------------------------------------------------------- pass 1
template <int KH>
__global__ void __launch_bounds__(kThreads, 1)
    score_stats_tc(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve<KH>(smem_raw, p);
    const uint32_t tmem = setup(s, p, 4);   // a slot is read by one warpgroup
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
        if (lane == 0) mma_issuer<KH, true>(s, p, tmem, t0, t1, nrb);
    } else {
        // Epilogue.  Warpgroup ewg owns the row blocks rb with rb % 2 == ewg;
        // a warp's TMEM lane quarter is fixed by its id % 4, so each thread
        // owns one query row per row block (two at most: m0/l0, m1/l1).
        const int quarter = warp & 3;
        const int ewg = (warp - 2) >> 2;
        const int row_in_blk = quarter * 32 + lane;
        float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
        uint32_t job = 0;
        bool ok = true;
        for (int64_t t = t0; t < t1 && ok; ++t) {
            const int u = (int)(t / p.tiles_per_unit);
            const int jt = (int)(t % p.tiles_per_unit);
            const int j0 = jt * kTileKeys;
            const bool last = (t == t1 - 1) || (jt == p.tiles_per_unit - 1);
            if (t == t0 || jt == 0) {
                m0 = m1 = -INFINITY;
                l0 = l1 = 0.f;
            }
            const bool masked = j0 + kTileKeys - 1 > p.P;
#pragma unroll 1
            for (int rb = ewg; rb < nrb; rb += 2) {
                const uint32_t jj = job + rb;
                const uint32_t slot = jj & 3, use = jj >> 2;
                if (!mbar_wait(&s.t_full[slot], use & 1, s.abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + slot * 128;
                const int r = rb * 128 + row_in_blk;
                // Largest column of this tile that row r may see.
                const int lim = masked ? p.P + (r % p.W) - j0 : kTileKeys - 1;
                float m = (rb >> 1) ? m1 : m0;
                float l = (rb >> 1) ? l1 : l0;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    float v[2][32];
                    load_row64(taddr + h * 64, v);
                    if (h == 1) release_slot(&s.t_empty[slot], lane);   // values are in registers
                    if (masked) {
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            if (h * 64 + i > lim) v[i >> 5][i & 31] = -INFINITY;
                    }
                    row_stats64_lazy(v, p.cs, m, l);
                }
                if (rb >> 1) {
                    m1 = m;
                    l1 = l;
                } else {
                    m0 = m;
                    l0 = l;
                }
            }
            job += nrb;
            if (!ok) break;
            if (last) {
                const int64_t slot_u = c - split_cta_of(p.n_tiles, p.grid, (int64_t)u * p.tiles_per_unit);
                float2 *dst = p.partial + ((int64_t)u * p.max_slots + slot_u) * p.rows_pad;
                for (int rb = ewg; rb < nrb; rb += 2) {
                    const int r = rb * 128 + row_in_blk;
                    if (r < p.rows) dst[r] = (rb >> 1) ? make_float2(m1, l1) : make_float2(m0, l0);
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
    const uint32_t tmem = setup(s, p, 8);   // both warpgroups read every slot
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c = blockIdx.x;
    const int64_t t0 = split_begin(p.n_tiles, p.grid, c), t1 = split_begin(p.n_tiles, p.grid, c + 1);
    const int nch = (p.n_pad + 255) / 256;   // query-row chunks of up to 256 (MMA N)

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            producer<KH>(s, p, &tq, &tk, t0, t1);
        }
    } else if (warp == 1) {
        if (lane == 0) mma_issuer<KH, false>(s, p, tmem, t0, t1, nch);
    } else {
        // Epilogue.  Each thread owns one key (its TMEM lane) and sums
        // 2^(x' * cs) over query rows, x' = q.k + nb_r / cs already in the
        // accumulator.  Every job (up to 256 rows) is split by columns:
        // warpgroup e reads columns [128 e, 128 e + 128), so a slot is free
        // again after two 64-column loads per warp; warpgroup 1 hands its
        // partial sum to warpgroup 0 through shared memory once per tile.
        const int quarter = warp & 3;
        const int ewg = (warp - 2) >> 2;
        const int etid = threadIdx.x - 64;
        const int key_in_tile = quarter * 32 + lane;
        const float rows_f = (float)p.rows;
        uint32_t job = 0, unit_changes = 0;
        bool ok = true;
        for (int64_t t = t0; t < t1 && ok; ++t) {
            const int u = (int)(t / p.tiles_per_unit);
            const int jt = (int)(t % p.tiles_per_unit);
            const int j0 = jt * kTileKeys;
            const uint32_t tl = (uint32_t)(t - t0);
            if (t == t0 || jt == 0) {
                // The unit's row biases become one more MMA K-step: row r of
                // aug_q holds nb_r / cs split into three bf16 terms (about 24
                // significant bits) in its first 16 bytes, zeros in the other
                // 16; every row of aug_k holds ones at the same three places in
                // both halves, so the product picks the terms up whatever the
                // 32-byte swizzle does to the two halves of a row.  Pad rows
                // get a bias that sends their exponentials to zero.
                if (unit_changes == 0) {
                    const __nv_bfloat16 one = __float2bfloat16(1.f), z = __float2bfloat16(0.f);
                    __align__(16) __nv_bfloat16 h8[8] = {one, one, one, z, z, z, z, z};
                    for (int i = etid; i < 128 * 2; i += kEpi)
                        *reinterpret_cast<uint4 *>(s.aug_k + i * 16) = *reinterpret_cast<const uint4 *>(h8);
                } else if (!mbar_wait(s.aug_empty, (unit_changes - 1) & 1, s.abort_flag, p.status)) {
                    break;   // the previous unit's MMAs still read aug_q
                }
                for (int r = etid; r < p.rows_pad; r += kEpi) {
                    const float nb = p.neg_bias_in[(int64_t)u * p.rows_pad + r];
                    const float v = (r < p.rows && nb > -3.0e4f * p.cs) ? nb / p.cs : -3.0e4f;
                    const __nv_bfloat16 hi = __float2bfloat16(v);
                    const float r1 = v - __bfloat162float(hi);
                    const __nv_bfloat16 mid = __float2bfloat16(r1);
                    const __nv_bfloat16 lo = __float2bfloat16(r1 - __bfloat162float(mid));
                    const __nv_bfloat16 z = __float2bfloat16(0.f);
                    __align__(16) __nv_bfloat16 h8[8] = {hi, mid, lo, z, z, z, z, z};
                    uint4 *dst = reinterpret_cast<uint4 *>(s.aug_q + (size_t)r * 32);
                    dst[0] = *reinterpret_cast<const uint4 *>(h8);
                    dst[1] = make_uint4(0u, 0u, 0u, 0u);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // visible to the MMA
                mbar_arrive(s.aug_full);
                ++unit_changes;
            }
            const int j = j0 + key_in_tile;
            const int dj = j - p.P;   // row r = g*W + w sees key j iff w >= dj
            const bool masked = j0 + kTileKeys - 1 > p.P;
            float a8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a8[i] = 0.f;
#pragma unroll 1
            for (int nc = 0; nc < nch; ++nc) {
                const uint32_t jj = job + nc;
                const uint32_t slot = jj & 1, use = jj >> 1;
                if (!mbar_wait(&s.t_full[slot], use & 1, s.abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int n = min(256, p.n_pad - nc * 256);
                const int c0 = ewg * 128;
                const int cn = min(128, n - c0);   // this warpgroup's columns (may be none)
                if (cn <= 0) {
                    release_slot(&s.t_empty[slot], lane);
                    continue;
                }
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + slot * 256 + c0;
                const int nh = (cn + 63) / 64;
#pragma unroll 1
                for (int h = 0; h < nh; ++h) {
                    float v[2][32];
                    load_row64(taddr + h * 64, v);
                    if (h == nh - 1) release_slot(&s.t_empty[slot], lane);
                    const int valid = cn - h * 64;   // narrow last chunk: 16..48 columns
                    if (valid < 64) {
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            if (i >= valid) v[i >> 5][i & 31] = -INFINITY;
                    }
                    if (masked) {
                        int w = (nc * 256 + c0 + h * 64) % p.W;
                        mask_cols(v[0], w, dj, p.W);
                        mask_cols(v[1], w, dj, p.W);
                    }
                    col_sums64(v, p.cs, a8);
                }
            }
            job += nch;
            if (!ok) break;
            float acc = ((a8[0] + a8[1]) + (a8[2] + a8[3])) + ((a8[4] + a8[5]) + (a8[6] + a8[7]));
            const uint32_t b = tl & 1, ub = tl >> 1;
            float *red = s.red + b * 128;
            if (ewg == 1) {
                if (!mbar_wait(&s.c_empty[b], (ub & 1) ^ 1, s.abort_flag, p.status)) break;
                red[key_in_tile] = acc;
                mbar_arrive(&s.c_full[b]);
            } else {
                if (!mbar_wait(&s.c_full[b], ub & 1, s.abort_flag, p.status)) break;
                acc += red[key_in_tile];
                mbar_arrive(&s.c_empty[b]);
                if (j < p.T) p.scores[(int64_t)u * p.T + j] = acc / rows_f;
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
