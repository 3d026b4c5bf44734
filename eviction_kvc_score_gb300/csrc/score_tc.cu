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
//   pass 1  D = Q K^T: each epilogue thread owns one TMEM lane = one query
//           row and keeps an online (max, sum) -> per-worker partials;
//   merge   (score_simt.cu) combines the partials into nb_r = -(m_r + log2 l_r);
//   pass 2  D = K Q^T plus one extra K-step that adds nb_r / (log2(e)/sqrt(D))
//           to every column r (ones against the row biases split into three
//           bf16 terms): each epilogue thread owns one key and sums
//           2^(x'_rj) over the query rows in registers -- no cross-lane
//           reduction in this orientation, and no per-logit bias load.
//
// Both passes run on SM pairs: a 2-CTA cluster issues cta_group::2 MMAs of
// M = 256 and N = 256 (measured on this GPU: 128 clk per 256x256x16 bf16
// MMA, the full rate of both SMs' tensor cores, against 166 clk for a
// single SM's 128x256x16 with both operands in shared memory).  The pair
// walks a contiguous run of (unit, 256-key tile) steps; CTA r of the pair
// holds keys [128 r, 128 r + 128) of each tile and the query row blocks
// [256 b + 128 r, +128) of the unit's Q block, which is exactly its share of
// the A and B operands in both orientations:
//   pass 1  A = Q rows (M = 256 over the pair), B = the tile's 256 keys;
//           CTA r's TMEM gets its 128 query rows x 256 keys;
//   pass 2  A = the tile's keys (M = 256), B = 256 query rows;
//           CTA r's TMEM gets its own 128 keys x 256 query rows.
// TMEM holds two 256-column accumulator slots (job b of a tile -> slot
// b mod 2).  Warp roles in each CTA: warp 0 TMA producer (its own K half and
// Q rows), warp 1 MMA issuer in the even CTA and, in the odd CTA, a relay
// that forwards each completed load to the even CTA's barriers; the other
// warps are the epilogue.  Pass 1 has four warpgroups, two per job of a tile,
// each folding 128 of the job's 256 key columns in two 64-column pieces (one
// job per warp and tile: the per-job waits, loads and bookkeeping are paid
// half as often as with every warpgroup reading every job).  Pass 2 has two
// warpgroups, each reading 128 columns of every job at once and freeing the
// slot before any arithmetic.  Each thread keeps independent sum chains on
// packed fp32 pairs; the window's causal mask sets invisible logits to -inf.
// Measured on this GPU, shared-memory loads in the epilogue compete with the
// MMAs' shared-memory operand reads, which is why pass 2 takes the row
// biases through the MMA; and every instruction per logit counts, which is
// why pass 1 keeps a running reference that is raised only when a piece
// would overflow instead of taking every piece's maximum.
//
// Keyformer (the NOISE instantiations; "Keyformer: KV Cache reduction
// through key tokens selection"): the same passes with logits
// (x_rj + zeta_rj) / tau, zeta the Gumbel draw of (unit, row, key) from
// Philox4x32-10 (kvc_internal.cuh, shared with the CUDA-core path), drawn in
// the epilogue for the visible logits only, 8 TMEM columns at a time; four
// epilogue warpgroups in both passes.
//
// Every wait is bounded (kvc_internal.cuh); there are no named barriers.
#include "kvc_internal.cuh"

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <cudaTypedefs.h>

namespace kvc {

namespace {

// Epilogue warpgroups per pass.  More warps hide more of the exponentials'
// latency, fewer carry less per-job overhead: pass 1 (a fold per row with a
// compare per piece) gains from four, pass 2 (a plain sum) runs best on two
// (measured on the 32K workload: four warpgroups there cost 4%).
constexpr int kEWG1 = 4, kEWG2 = 2;
constexpr int kMaxEWG = 4;
__host__ __device__ constexpr int wg_cols(int ewg) { return 256 / ewg; }   // columns per warpgroup
__host__ __device__ constexpr int epi_threads(int ewg) { return 128 * ewg; }
__host__ __device__ constexpr int cta_threads(int ewg) { return 64 + epi_threads(ewg); }
// Registers per thread: each of the SM's four schedulers has a quarter of
// the register file for the warps it holds (warps are dealt round-robin), in
// steps of 8 per thread.
__host__ __device__ constexpr int max_regs(int ewg) {
    return (16384 / (((cta_threads(ewg) / 32 + 3) / 4) * 32)) / 8 * 8;
}
constexpr uint32_t kTmemCols = 512;
constexpr int kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 64 bf16
constexpr int kSlotCols = 256;        // TMEM columns per accumulator slot
constexpr int kMinSmem = 120 * 1024;  // > half an SM's shared memory: one CTA per SM
constexpr int kRedBytes = (kMaxEWG - 1) * 2 * 128 * 8;   // epilogue hand-over buffer

struct TcParams {
    int64_t n_tiles;          // (unit, 256-key tile) steps
    int64_t tiles_per_unit;
    int pairs;
    int max_slots;
    int T, P, W;
    int rows;       // G*W
    int rows_pad;   // multiple of 256
    int rows_half;  // rows_pad / 2: query rows held by one CTA
    int stages;
    float cs;       // log2(e) / (sqrt(D) tau); tau = 1 without noise
    float noise_scale;      // log2(e) / tau (Keyformer noise)
    uint32_t key0, key1;    // Philox key (Keyformer noise)
    int skip_first_relay;   // test knob: the odd CTA withholds its first load's arrival
    float2 *partial;
    const float *neg_bias_in;
    float *scores;
    uint32_t *status;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Shared-memory carve-up, identical in both CTAs of a pair (the MMA reads
// the odd CTA's operands at the even CTA's offsets).
struct Smem {
    uint8_t *q;        // [KH][rows_half][128 B], 128-byte swizzled (TMA)
    uint8_t *k;        // [stages][KH][128 keys][128 B]
    uint8_t *aug_k;    // [128 keys][32 B] pass-2 extra K-step operand: ones
    uint8_t *aug_q;    // [rows_half][32 B] pass-2 extra K-step operand: row biases
    float2 *red;       // epilogue hand-over warpgroups 1.. -> 0 (kRedBytes)
    uint64_t *full, *empty, *pfull;   // K ring: own loads, MMA done, peer's loads (even CTA)
    uint64_t *q_full, *q_empty, *q_pfull;
    uint64_t *t_full, *t_empty;       // [2] TMEM slots (t_empty counts both CTAs' warps)
    uint64_t *c_full, *c_empty;       // [2]
    uint64_t *aug_full, *aug_empty, *drain;
    uint32_t *tmem_base;
    volatile int *abort_flag;
};

template <int KH>
__device__ __forceinline__ Smem carve(uint8_t *raw, const TcParams &p) {
    Smem s;
    uint8_t *b = align1024(raw);
    s.q = b;
    b += (size_t)KH * p.rows_half * 128;
    s.k = b;
    b += (size_t)p.stages * KH * kBoxBytes;
    s.aug_k = b;
    b += 128 * 32;
    s.aug_q = b;
    b += (size_t)p.rows_half * 32;
    s.red = reinterpret_cast<float2 *>(b);
    b += kRedBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(b);
    s.full = bars;
    s.empty = bars + p.stages;
    s.pfull = bars + 2 * p.stages;
    s.q_full = bars + 3 * p.stages;
    s.q_empty = s.q_full + 1;
    s.q_pfull = s.q_empty + 1;
    s.t_full = s.q_pfull + 1;   // 2
    s.t_empty = s.t_full + 2;   // 2
    s.c_full = s.t_empty + 2;   // 2
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
    const size_t need = 1024 + (size_t)KH * (rows_pad / 2) * 128 + (size_t)stages * KH * kBoxBytes +
                        128 * 32 + (size_t)(rows_pad / 2) * 32 + kRedBytes +
                        (size_t)(3 * stages + 14) * 8 + 16;
    return need < (size_t)kMinSmem ? (size_t)kMinSmem : need;
}

// (unit, tile) of step t, kept incrementally: no 64-bit division per step.
struct Step {
    int u, jt, tpu;
    __device__ Step(int64_t t, int64_t tiles_per_unit)
        : u((int)(t / tiles_per_unit)), jt((int)(t % tiles_per_unit)), tpu((int)tiles_per_unit) {}
    __device__ void next() {
        if (++jt == tpu) {
            jt = 0;
            ++u;
        }
    }
};

// Barrier set-up and TMEM allocation in both CTAs; returns the TMEM base.
template <int EWG>
__device__ __forceinline__ uint32_t setup(const Smem &s, const TcParams &p, uint32_t t_empty_count,
                                          uint32_t c_full_count) {
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
            mbar_init(&s.pfull[i], 1);
        }
        mbar_init(s.q_full, 1);
        mbar_init(s.q_empty, 1);
        mbar_init(s.q_pfull, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.t_full[i], 1);
            mbar_init(&s.t_empty[i], t_empty_count);   // epilogue warps of both CTAs
            mbar_init(&s.c_full[i], c_full_count);
            mbar_init(&s.c_empty[i], 128);
        }
        mbar_init(s.aug_full, 2 * epi_threads(EWG));
        mbar_init(s.aug_empty, 1);
        mbar_init(s.drain, 1);
        *s.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc2(s.tmem_base, kTmemCols);
        tmem_relinquish2();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // the peer's barriers exist before any remote arrive
    tc_fence_after();
    return *s.tmem_base;
}

__device__ __forceinline__ void teardown(uint32_t tmem) {
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // no MMA, load or remote arrive of the pair is left
    if ((threadIdx.x >> 5) == 1) {
        tc_fence_after();
        tmem_dealloc2(tmem, kTmemCols);
    }
    cluster_sync_all();
}

// TMA producer (one thread per CTA): the CTA's Q rows whenever the unit
// changes, then its 128-key half of each tile.  Returns after draining its
// own copies.
template <int KH>
__device__ void producer(const Smem &s, const TcParams &p, const CUtensorMap *tq,
                         const CUtensorMap *tk, int64_t t0, int64_t t1, int rank) {
    int stage = 0;
    uint32_t phase = 0;
    uint32_t q_loads = 0;
    int64_t issued = 0;
    Step st(t0, p.tiles_per_unit);
    for (int64_t t = t0; t < t1; ++t, st.next()) {
        const int u = st.u, jt = st.jt;
        if (t == t0 || jt == 0) {
            if (q_loads > 0 && !mbar_wait(s.q_empty, (q_loads - 1) & 1, s.abort_flag, p.status))
                break;
            mbar_arrive_expect_tx(s.q_full, (uint32_t)(KH * p.rows_half * 128));
            for (int kh = 0; kh < KH; ++kh)
                for (int b = 0; b < p.rows_half / 128; ++b)
                    tma_load_3d(tq, s.q_full, s.q + ((size_t)kh * p.rows_half + b * 128) * 128,
                                kh * 64, b * 256 + rank * 128, u);
            ++q_loads;
        }
        if (!mbar_wait(&s.empty[stage], phase ^ 1, s.abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&s.full[stage], (uint32_t)(KH * kBoxBytes));
        for (int kh = 0; kh < KH; ++kh)
            tma_load_3d(tk, &s.full[stage], s.k + ((size_t)stage * KH + kh) * kBoxBytes, kh * 64,
                        jt * kPairKeys + rank * 128, u);
        ++issued;
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1;
        }
    }
    // Unwind: every copy this thread started must land before the CTA exits.
    if (*s.abort_flag) {
        for (int64_t i = issued > p.stages ? issued - p.stages : 0; i < issued; ++i)
            mbar_drain(&s.full[i % p.stages], (uint32_t)((i / p.stages) & 1));
        if (q_loads > 0) mbar_drain(s.q_full, (q_loads - 1) & 1);
    }
}

// Odd CTA (one thread): forward the completion of each of its own loads to
// the even CTA, whose MMAs read them.
__device__ void relay(const Smem &s, const TcParams &p, int64_t t0, int64_t t1) {
    const uint32_t r_pfull = mapa_shared(smem_u32(s.pfull), 0);
    const uint32_t r_qpfull = mapa_shared(smem_u32(s.q_pfull), 0);
    int stage = 0;
    uint32_t phase = 0, q_loads = 0;
    Step st(t0, p.tiles_per_unit);
    for (int64_t t = t0; t < t1; ++t, st.next()) {
        const int jt = st.jt;
        if (t == t0 || jt == 0) {
            if (!mbar_wait(s.q_full, q_loads & 1, s.abort_flag, p.status)) break;
            mbar_arrive_remote(r_qpfull);
            ++q_loads;
        }
        if (!mbar_wait(&s.full[stage], phase, s.abort_flag, p.status)) break;
        // (the test knob leaves the even CTA waiting for this arrival: its
        // bounded wait runs out, it records KVC_DEV_TIMEOUT and the pair
        // unwinds)
        if (!(p.skip_first_relay && t == t0)) mbar_arrive_remote(r_pfull + (uint32_t)stage * 8u);
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1;
        }
    }
}

__device__ __forceinline__ void mma_drain(const Smem &s) {
    tc_commit2(s.drain, 1);
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

// MMA issuer (one thread of the even CTA).  For every tile: njob jobs of
// 256 x 256 fp32 accumulators into slot job % 2 of both CTAs' TMEM.
// Pass 1 (KEYS_AS_B): A = Q rows of job b (each CTA's local block b), B = the
// tile's keys.  Pass 2: A = the tile's keys, B = Q rows of job b, then the
// bias K-step.
template <int KH, bool KEYS_AS_B>
__device__ void mma_issuer(const Smem &s, const TcParams &p, uint32_t tmem, int64_t t0, int64_t t1,
                           int njob) {
    constexpr uint16_t kBoth = 3;
    const uint32_t idesc = idesc_bf16_f32(256, 256);
    int stage = 0;
    uint32_t phase = 0, q_loads = 0, job = 0;
    bool ok = true;
    Step st(t0, p.tiles_per_unit);
    for (int64_t t = t0; t < t1 && ok; ++t, st.next()) {
        const int jt = st.jt;
        const bool last = (t == t1 - 1) || (jt == p.tiles_per_unit - 1);
        if (t == t0 || jt == 0) {
            if (!mbar_wait(s.q_full, q_loads & 1, s.abort_flag, p.status)) break;
            if (!mbar_wait(s.q_pfull, q_loads & 1, s.abort_flag, p.status)) break;
            // pass 2 also needs both CTAs' row-bias operands for the unit
            if (!KEYS_AS_B && !mbar_wait_cl(s.aug_full, q_loads & 1, s.abort_flag, p.status)) break;
            ++q_loads;
        }
        if (!mbar_wait(&s.full[stage], phase, s.abort_flag, p.status)) break;
        if (!mbar_wait(&s.pfull[stage], phase, s.abort_flag, p.status)) break;
        tc_fence_after();
        for (int jb = 0; jb < njob; ++jb, ++job) {
            const uint32_t slot = job & 1, use = job >> 1;
            if (!mbar_wait(&s.t_empty[slot], (use & 1) ^ 1, s.abort_flag, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + slot * kSlotCols;
            // one descriptor per operand and job; a K-step only moves the
            // start address field (16-byte units): -1% of kvc_score at 32K
            const uint64_t qd = sw128_kmajor_desc(smem_u32(s.q + (size_t)jb * 128 * 128));
            const uint64_t kd = sw128_kmajor_desc(smem_u32(s.k + (size_t)stage * KH * kBoxBytes));
#pragma unroll
            for (int ks = 0; ks < KH * 4; ++ks) {
                const int kh = ks >> 2, off = (ks & 3) * 32;
                const uint64_t qs = qd + (uint64_t)(((size_t)kh * p.rows_half * 128 + off) >> 4);
                const uint64_t kk = kd + (uint64_t)((kh * kBoxBytes + off) >> 4);
                tc_mma2_bf16(d, KEYS_AS_B ? qs : kk, KEYS_AS_B ? kk : qs, idesc, ks > 0);
            }
            if (!KEYS_AS_B) {
                // one more K-step adds each query row's bias to its column:
                // ones (keys) x the row's bias / cs split into bf16 terms
                tc_mma2_bf16(d, sw32_kmajor_desc(smem_u32(s.aug_k)),
                             sw32_kmajor_desc(smem_u32(s.aug_q + (size_t)jb * 128 * 32)), idesc, 1u);
            }
            tc_commit2(&s.t_full[slot], kBoth);
        }
        if (!ok) break;
        tc_commit2(&s.empty[stage], kBoth);
        if (last) tc_commit2(s.q_empty, kBoth);
        if (last && !KEYS_AS_B) tc_commit2(s.aug_empty, kBoth);
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1;
        }
    }
    mma_drain(s);
}

// Release a TMEM slot (on the even CTA's barrier) once this warp's loads
// from it have completed.
__device__ __forceinline__ void release_slot(uint32_t r_bar, int lane) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_remote(r_bar);
}

// 32 NC consecutive fp32 columns of this thread's TMEM lane -> v, completed
// (all loads in flight, one wait): the warp's whole share of a slot, so the
// slot can be released before any arithmetic.
template <int NC>
__device__ __forceinline__ void load_cols(uint32_t taddr, float (&v)[NC][32]) {
#pragma unroll
    for (int i = 0; i < NC; ++i) tmem_ld32(taddr + 32 * i, v[i]);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < NC; ++i) reg_fence(v[i]);
}
// 8 consecutive fp32 columns -> v, completed.
__device__ __forceinline__ void load_cols8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
    tmem_ld_wait();
    asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// The 64-column piece h of a row.
template <int NC>
__device__ __forceinline__ float (&piece64(float (&v)[NC][32], int h))[2][32] {
    return *reinterpret_cast<float(*)[2][32]>(&v[2 * h]);
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
// The exact fold (a row's first piece, or a piece that would overflow) is
// one shared code path: a second inlined copy cost registers and ~1% of
// pass 1.
__device__ __forceinline__ void row_stats64_lazy(const float (&v)[2][32], float cs, float &m_run,
                                                 float &l_run) {
    if (m_run != -INFINITY) {
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
    }
    // first piece of a row, or one that would overflow: fold exactly
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

// v[base + s] for a run-time s in 0..3 (selects, no local memory).
__device__ __forceinline__ float pick4f(const float (&v)[8], int base, int s) {
    const float a = (s & 1) ? v[base + 1] : v[base], b = (s & 1) ? v[base + 3] : v[base + 2];
    return (s & 2) ? b : a;
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

// Combine two (max, sum) folds of the same row: l * 2^m is the sum either way.
__device__ __forceinline__ void fold_pair(float &m, float &l, float2 o) {
    if (o.x == -INFINITY) return;
    if (m == -INFINITY) {
        m = o.x;
        l = o.y;
        return;
    }
    const float mn = fmaxf(m, o.x);
    l = l * ex2(m - mn) + o.y * ex2(o.x - mn);
    m = mn;
}

// --------------------------------------------------------------- pass 1
template <int KH, int EWG, bool NOISE>
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(max_regs(EWG))
    score_stats_tc(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve<KH>(smem_raw, p);
    const int njob = p.rows_pad / 256;
    const int wpj = EWG / njob;   // epilogue warpgroups per job
    // a slot is read by the job's warpgroups in both CTAs; the other
    // warpgroups of a job hand their folds to its first one
    const uint32_t tmem =
        setup<EWG>(s, p, 2u * 4u * wpj, wpj > 1 ? (uint32_t)(wpj - 1) * 128u : 1u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)cluster_ctarank();
    const int64_t c = cluster_id_x();
    const int64_t t0 = split_begin(p.n_tiles, p.pairs, c), t1 = split_begin(p.n_tiles, p.pairs, c + 1);

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            producer<KH>(s, p, &tq, &tk, t0, t1, rank);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            if (rank == 0)
                mma_issuer<KH, true>(s, p, tmem, t0, t1, njob);
            else
                relay(s, p, t0, t1);
        }
    } else {
        // Epilogue.  The warpgroups are split between the tile's jobs: wpj =
        // EWG / njob of them read job my_job, warpgroup sub of those the key
        // columns [cols sub, +cols) in 64-column pieces.  A warp's TMEM lane
        // quarter is fixed by its id % 4, so each thread owns query row
        // 256 my_job + 128 rank + 32 quarter + lane over its share of the
        // tile's keys; the shares of a row are combined when the unit ends,
        // in warpgroup order.
        const int quarter = warp & 3;
        const int ewg = (warp - 2) >> 2;
        const int row_in_blk = quarter * 32 + lane;
        const int my_job = ewg / wpj, sub = ewg % wpj;
        const int cols = kPairKeys / wpj, npc = cols / 64;
        const int r = my_job * 256 + rank * 128 + row_in_blk;
        const bool pad = my_job * 256 + rank * 128 >= p.rows;   // this CTA's rows of the job
        const int w_r = r % p.W;                                 // window position of row r
        const uint32_t r_tempty = mapa_shared(smem_u32(s.t_empty), 0);
        float m = -INFINITY, l = 0.f;
        uint32_t job = 0, unit_ends = 0;
        bool ok = true;
        Step st(t0, p.tiles_per_unit);
        for (int64_t t = t0; t < t1 && ok; ++t, st.next()) {
            const int u = st.u, jt = st.jt;
            const int j0 = jt * kPairKeys + sub * cols;   // this warpgroup's first key
            const bool last = (t == t1 - 1) || (jt == p.tiles_per_unit - 1);
            if (t == t0 || jt == 0) {
                m = -INFINITY;
                l = 0.f;
            }
            const bool masked = j0 + cols - 1 > p.P;
            const uint32_t jj = job + my_job;
            const uint32_t slot = jj & 1, use = jj >> 1;
            job += njob;
            if (!mbar_wait(&s.t_full[slot], use & 1, s.abort_flag, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t taddr =
                tmem + ((uint32_t)(quarter * 32) << 16) + slot * kSlotCols + sub * cols;
            if (pad) {
                release_slot(r_tempty + slot * 8u, lane);
            } else if constexpr (NOISE) {
                // Keyformer: base-2 noisy logits x cs + zeta log2(e)/tau (the
                // Gumbel draw of (unit, row, key)), drawn only where the row
                // sees the key, folded exactly 8 columns at a time
                const int lim = masked ? p.P + w_r - j0 : cols - 1;
#pragma unroll 1
                for (int ch = 0; ch < cols / 8; ++ch) {
                    float v8[8];
                    load_cols8(taddr + ch * 8, v8);
                    if (ch == cols / 8 - 1) release_slot(r_tempty + slot * 8u, lane);
                    // the chunk's 8 keys are two whole Philox blocks of row r
                    uint32_t w[2][4];
                    const uint32_t blk = (uint32_t)(j0 + ch * 8) >> 2;
                    philox4(blk, (uint32_t)r, (uint32_t)u, p.key0, p.key1, w[0]);
                    philox4(blk + 1u, (uint32_t)r, (uint32_t)u, p.key0, p.key1, w[1]);
                    float mx = -INFINITY;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int col = ch * 8 + i;
                        v8[i] = col <= lim ? fmaf(gumbel_bits(w[i >> 2][i & 3]), p.noise_scale,
                                                  v8[i] * p.cs)
                                           : -INFINITY;
                        mx = fmaxf(mx, v8[i]);
                    }
                    if (mx > -INFINITY) {
                        const float mnew = fmaxf(m, mx);
                        float sum = 0.f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) sum += ex2(v8[i] - mnew);
                        l = l * ex2(m - mnew) + sum;
                        m = mnew;
                    }
                }
            } else {
                // Largest column of this warpgroup's share that row r may see.
                const int lim = masked ? p.P + w_r - j0 : cols - 1;
#pragma unroll 1
                for (int h = 0; h < npc; ++h) {
                    float v[2][32];
                    load_cols(taddr + h * 64, v);
                    if (h == npc - 1) release_slot(r_tempty + slot * 8u, lane);
                    if (masked) {
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            if (h * 64 + i > lim) v[i >> 5][i & 31] = -INFINITY;
                    }
                    row_stats64_lazy(v, p.cs, m, l);
                }
            }
            if (last) {
                const uint32_t ue = unit_ends++;
                float2 *red = s.red + my_job * (kMaxEWG - 1) * 128;
                if (sub > 0) {
                    if (!mbar_wait(&s.c_empty[my_job], (ue & 1) ^ 1, s.abort_flag, p.status)) break;
                    red[(sub - 1) * 128 + row_in_blk] = make_float2(m, l);
                    mbar_arrive(&s.c_full[my_job]);
                } else {
                    if (wpj > 1) {   // a job with one warpgroup has nothing to combine
                        if (!mbar_wait(&s.c_full[my_job], ue & 1, s.abort_flag, p.status)) break;
                        for (int e = 1; e < wpj; ++e)
                            fold_pair(m, l, red[(e - 1) * 128 + row_in_blk]);
                        mbar_arrive(&s.c_empty[my_job]);
                    }
                    const int64_t slot_u =
                        c - split_cta_of(p.n_tiles, p.pairs, (int64_t)u * p.tiles_per_unit);
                    float2 *dst = p.partial + ((int64_t)u * p.max_slots + slot_u) * p.rows_pad;
                    if (r < p.rows) dst[r] = make_float2(m, l);
                }
            }
        }
    }
    teardown(tmem);
}

// --------------------------------------------------------------- pass 2
template <int KH, int EWG, bool NOISE>
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(max_regs(EWG))
    score_colmean_tc(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve<KH>(smem_raw, p);
    const uint32_t tmem = setup<EWG>(s, p, 2u * 4u * EWG, (uint32_t)(EWG - 1) * 128u);
    constexpr int kCols = wg_cols(EWG);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)cluster_ctarank();
    const int64_t c = cluster_id_x();
    const int64_t t0 = split_begin(p.n_tiles, p.pairs, c), t1 = split_begin(p.n_tiles, p.pairs, c + 1);
    const int njob = p.rows_pad / 256;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            producer<KH>(s, p, &tq, &tk, t0, t1, rank);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            if (rank == 0)
                mma_issuer<KH, false>(s, p, tmem, t0, t1, njob);
            else
                relay(s, p, t0, t1);
        }
    } else {
        // Epilogue.  Each thread owns one of the CTA's keys (its TMEM lane)
        // and sums 2^(x' * cs) over query rows, x' = q.k + nb_r / cs already
        // in the accumulator.  Warpgroup e reads columns [kCols e, +kCols)
        // of every job (query rows 256 b + kCols e + i); warpgroups 1.. hand
        // their partial sums to warpgroup 0 through shared memory once per
        // tile, added in warpgroup order.
        const int quarter = warp & 3;
        const int ewg = (warp - 2) >> 2;
        const int etid = threadIdx.x - 64;
        const int key_in_tile = quarter * 32 + lane;
        const float rows_f = (float)p.rows;
        const uint32_t r_tempty = mapa_shared(smem_u32(s.t_empty), 0);
        const uint32_t r_augfull = mapa_shared(smem_u32(s.aug_full), 0);
        float *red = reinterpret_cast<float *>(s.red);
        uint32_t job = 0, unit_changes = 0;
        bool ok = true;
        Step st(t0, p.tiles_per_unit);
        for (int64_t t = t0; t < t1 && ok; ++t, st.next()) {
            const int u = st.u, jt = st.jt;
            const int j0 = jt * kPairKeys + rank * 128;   // this CTA's first key
            const uint32_t tl = (uint32_t)(t - t0);
            if (t == t0 || jt == 0) {
                // The unit's row biases become one more MMA K-step: local row
                // i of aug_q (query row 256 (i / 128) + 128 rank + i % 128)
                // holds nb_r / cs split into three bf16 terms (about 24
                // significant bits) in its first 16 bytes, zeros in the other
                // 16; every row of aug_k holds ones at the same three places in
                // both halves, so the product picks the terms up whatever the
                // 32-byte swizzle does to the two halves of a row.  Pad rows
                // get a bias that sends their exponentials to zero.
                if (unit_changes == 0) {
                    const __nv_bfloat16 one = __float2bfloat16(1.f), z = __float2bfloat16(0.f);
                    __align__(16) __nv_bfloat16 h8[8] = {one, one, one, z, z, z, z, z};
                    for (int i = etid; i < 128 * 2; i += epi_threads(EWG))
                        *reinterpret_cast<uint4 *>(s.aug_k + i * 16) = *reinterpret_cast<const uint4 *>(h8);
                } else if (!mbar_wait(s.aug_empty, (unit_changes - 1) & 1, s.abort_flag, p.status)) {
                    break;   // the previous unit's MMAs still read aug_q
                }
                for (int i = etid; i < p.rows_half; i += epi_threads(EWG)) {
                    const int r = (i >> 7) * 256 + rank * 128 + (i & 127);
                    const float nb = p.neg_bias_in[(int64_t)u * p.rows_pad + r];
                    const float v = (r < p.rows && nb > -3.0e4f * p.cs) ? nb / p.cs : -3.0e4f;
                    const __nv_bfloat16 hi = __float2bfloat16(v);
                    const float r1 = v - __bfloat162float(hi);
                    const __nv_bfloat16 mid = __float2bfloat16(r1);
                    const __nv_bfloat16 lo = __float2bfloat16(r1 - __bfloat162float(mid));
                    const __nv_bfloat16 z = __float2bfloat16(0.f);
                    __align__(16) __nv_bfloat16 h8[8] = {hi, mid, lo, z, z, z, z, z};
                    uint4 *dst = reinterpret_cast<uint4 *>(s.aug_q + (size_t)i * 32);
                    dst[0] = *reinterpret_cast<const uint4 *>(h8);
                    dst[1] = make_uint4(0u, 0u, 0u, 0u);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // visible to the MMA
                mbar_arrive_remote_cluster(r_augfull);
                ++unit_changes;
            }
            const int j = j0 + key_in_tile;
            const int dj = j - p.P;   // row r = g*W + w sees key j iff w >= dj
            const bool masked = j0 + 127 > p.P;   // this CTA's 128 keys reach the window
            float a8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a8[i] = 0.f;
#pragma unroll 1
            for (int nc = 0; nc < njob; ++nc) {
                const uint32_t jj = job + nc;
                const uint32_t slot = jj & 1, use = jj >> 1;
                if (!mbar_wait(&s.t_full[slot], use & 1, s.abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int n = min(256, p.rows - nc * 256);   // real query rows of this job
                const int c0 = ewg * kCols;
                const int cn = min(kCols, n - c0);   // this warpgroup's columns (may be none)
                if (cn <= 0) {
                    release_slot(r_tempty + slot * 8u, lane);
                    continue;
                }
                if constexpr (NOISE) {
                    // Keyformer: 2^(x' cs + zeta log2(e)/tau) over the rows
                    // that see this key, 8 columns at a time
                    const uint32_t taddr8 =
                        tmem + ((uint32_t)(quarter * 32) << 16) + slot * kSlotCols + c0;
                    const int nch = (cn + 7) / 8;
                    // Draws: the four lanes of a key block (keys 4m..4m+3, m =
                    // j / 4) each compute the Philox block of one of four rows,
                    // then a 4 x 4 transpose by xor-shuffles hands every lane
                    // its own key's word of each row: in round x lane b sends
                    // word b ^ x and receives, from lane b ^ x, its key's word
                    // of row b ^ x.
                    const uint32_t bq = (uint32_t)lane & 3u;
#pragma unroll 1
                    for (int ch = 0; ch < nch; ++ch) {
                        float v8[8];
                        load_cols8(taddr8 + ch * 8, v8);
                        if (ch == nch - 1) release_slot(r_tempty + slot * 8u, lane);
                        const int row0 = nc * 256 + c0 + ch * 8;   // rows row0 .. row0 + 7
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            uint32_t w[4];
                            philox4((uint32_t)j >> 2, (uint32_t)(row0 + 4 * c) + bq, (uint32_t)u,
                                    p.key0, p.key1, w);
#pragma unroll
                            for (int x = 0; x < 4; ++x) {
                                const uint32_t send = pick4(w, bq ^ (uint32_t)x);
                                const uint32_t got =
                                    x == 0 ? send : __shfl_xor_sync(0xffffffffu, send, x);
                                const int i = 4 * c + (int)(bq ^ (uint32_t)x);   // this draw's column
                                const float vi = (i & 4) ? pick4f(v8, 4, i & 3) : pick4f(v8, 0, i & 3);
                                const int row = row0 + i;
                                const bool vis = ch * 8 + i < cn && (!masked || row % p.W >= dj);
                                if (vis)
                                    a8[4 * c + x] += ex2(fmaf(gumbel_bits(got), p.noise_scale,
                                                              vi * p.cs));
                            }
                        }
                    }
                    continue;
                }
                const uint32_t taddr =
                    tmem + ((uint32_t)(quarter * 32) << 16) + slot * kSlotCols + c0;
                float v[kCols / 32][32];
                load_cols(taddr, v);
                release_slot(r_tempty + slot * 8u, lane);   // values are in registers
                if (cn < kCols) {   // narrow last job: columns past the real rows
#pragma unroll
                    for (int i = 0; i < kCols; ++i)
                        if (i >= cn) v[i >> 5][i & 31] = -INFINITY;
                }
                if (masked) {
                    int w = (nc * 256 + c0) % p.W;
#pragma unroll
                    for (int q = 0; q < kCols / 32; ++q) mask_cols(v[q], w, dj, p.W);
                }
#pragma unroll
                for (int h = 0; h < kCols / 64; ++h)
                    if (cn > 64 * h) col_sums64(piece64(v, h), p.cs, a8);
            }
            job += njob;
            if (!ok) break;
            float acc = ((a8[0] + a8[1]) + (a8[2] + a8[3])) + ((a8[4] + a8[5]) + (a8[6] + a8[7]));
            const uint32_t b = tl & 1, ub = tl >> 1;
            float *rb = red + b * (EWG - 1) * 128;
            if (ewg > 0) {
                if (!mbar_wait(&s.c_empty[b], (ub & 1) ^ 1, s.abort_flag, p.status)) break;
                rb[(ewg - 1) * 128 + key_in_tile] = acc;
                mbar_arrive(&s.c_full[b]);
            } else {
                if (!mbar_wait(&s.c_full[b], ub & 1, s.abort_flag, p.status)) break;
#pragma unroll
                for (int e = 0; e < EWG - 1; ++e) acc += rb[e * 128 + key_in_tile];
                mbar_arrive(&s.c_empty[b]);
                if (j < p.T) p.scores[(int64_t)u * p.T + j] = acc / rows_f;
            }
        }
    }
    teardown(tmem);
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

}  // namespace

bool make_tma_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t mid, uint64_t outer,
                  uint32_t box_rows) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {inner, mid, outer};
    cuuint64_t strides[2] = {inner * 2, inner * mid * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

// 3-D bf16 view [outer][mid][inner] with a (64, 128, 1) box, 128-byte swizzle.
// Rows past `mid` read as zeros.
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t mid, uint64_t outer) {
    return make_tma_map(m, base, inner, mid, outer, 128);
}

constexpr size_t kSmemLimit = 232448;   // 227 KiB per CTA

template <int KH>
int pick_stages(int rows_pad) {
    // Deepest K ring that fits next to the resident Q rows.
    int stages = 4;
    while (stages > 2 && smem_bytes<KH>(rows_pad, stages) > kSmemLimit) --stages;
    return stages;
}

// Keyformer's noise makes the epilogue ALU-bound (a Philox draw and two
// logarithms per logit): four warpgroups in both passes hide the draws'
// dependency chains better than two (measured 0.77 vs 1.20 ms on one 16K
// Llama-3-8B-shaped layer).
constexpr int kEWGNoise = 4;

template <int KH>
void set_smem_attr() {
    static bool done = false;
    if (!done) {
        cudaFuncSetAttribute(score_stats_tc<KH, kEWG1, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
        cudaFuncSetAttribute(score_colmean_tc<KH, kEWG2, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
        cudaFuncSetAttribute(score_stats_tc<KH, kEWGNoise, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
        cudaFuncSetAttribute(score_colmean_tc<KH, kEWGNoise, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
        done = true;
    }
}

template <int KH>
int launch_kh(const kvc_shape &s, const ScoreSplit &sp, const ScoreArgs &a, cudaStream_t st,
              bool noise, uint64_t seed, double tau) {
    const int G = s.n_q_heads / s.n_kv_heads;
    CUtensorMap tq, tk;
    if (!make_map(&tq, a.q, (uint64_t)s.head_dim, (uint64_t)G * s.window, (uint64_t)sp.n_units) ||
        !make_map(&tk, a.k, (uint64_t)s.head_dim, (uint64_t)s.seq_len, (uint64_t)sp.n_units)) {
        set_error("kvc_score: cuTensorMapEncodeTiled failed (alignment or driver)");
        return KVC_ERR_CUDA;
    }
    if (sp.rows_pad % 256 || sp.rows_pad > kMaxRowsTC) {
        set_error("kvc_score: tensor-core split needs rows padded to 256 (got %d)", sp.rows_pad);
        return KVC_ERR_UNSUPPORTED;
    }
    TcParams p;
    p.n_tiles = sp.n_tiles;
    p.tiles_per_unit = sp.tiles_per_unit;
    p.pairs = sp.grid;
    p.max_slots = sp.max_slots;
    p.T = s.seq_len;
    p.W = s.window;
    p.P = s.seq_len - s.window;
    p.rows = sp.rows;
    p.rows_pad = sp.rows_pad;
    p.rows_half = sp.rows_pad / 2;
    // Keyformer divides the noisy logits by tau: both the logit scale and
    // the noise scale carry 1/tau (plain scores: tau = 1, no noise)
    p.cs = (float)(kLog2e / sqrt((double)s.head_dim) / tau);
    p.noise_scale = (float)(kLog2e / tau);
    p.key0 = (uint32_t)seed;
    p.key1 = (uint32_t)(seed >> 32);
    p.partial = a.partial;
    p.neg_bias_in = a.neg_bias;
    p.scores = a.scores;
    p.status = a.status;
    // Test knob (KVC_TEST_SKIP_ARRIVE=1): pass 1 runs with one arrival
    // withheld, so every pair's bounded waits run out; used only to check
    // that the timeout is reported and the context stays usable.
    const char *skip = getenv("KVC_TEST_SKIP_ARRIVE");
    p.skip_first_relay = (skip && skip[0] == '1') ? 1 : 0;
    p.stages = pick_stages<KH>(sp.rows_pad);
    const size_t smem = smem_bytes<KH>(sp.rows_pad, p.stages);
    set_smem_attr<KH>();
    const int ctas = 2 * sp.grid;   // one 2-CTA cluster per pair
    if (noise)
        score_stats_tc<KH, kEWGNoise, true><<<ctas, cta_threads(kEWGNoise), smem, st>>>(tq, tk, p);
    else
        score_stats_tc<KH, kEWG1, false><<<ctas, cta_threads(kEWG1), smem, st>>>(tq, tk, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_score: pass-1 launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    int rc = launch_score_merge(s, sp, a, st);
    if (rc || a.stats_only) return rc;
    p.skip_first_relay = 0;
    if (noise)
        score_colmean_tc<KH, kEWGNoise, true><<<ctas, cta_threads(kEWGNoise), smem, st>>>(tq, tk, p);
    else
        score_colmean_tc<KH, kEWG2, false><<<ctas, cta_threads(kEWG2), smem, st>>>(tq, tk, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_score: pass-2 launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

}  // namespace

int score_tc_pairs(int sms) {
    constexpr int kMaxDev = 64;
    static int cached[kMaxDev] = {0};
    int dev = 0;
    const int fallback = (sms > 0 ? sms : 148) / 2;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
        cudaGetLastError();
        return fallback;
    }
    if (cached[dev]) return cached[dev];
    // Clusters of the largest configuration (head_dim 128, 512 rows) that
    // the device keeps resident at once: a persistent grid larger than that
    // would run its last pairs in a second wave.
    int n = fallback;
    set_smem_attr<2>();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * fallback, 1, 1);
    cfg.blockDim = dim3(cta_threads(kEWG1), 1, 1);
    cfg.dynamicSmemBytes = smem_bytes<2>(kMaxRowsTC, pick_stages<2>(kMaxRowsTC));
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, score_stats_tc<2, kEWG1, false>, &cfg) ==
            cudaSuccess &&
        clusters > 0) {
        if (clusters < n) n = clusters;
    } else {
        cudaGetLastError();
    }
    cached[dev] = n;
    return n;
}

int launch_score_tc(const kvc_shape &s, const ScoreSplit &sp, const ScoreArgs &a, cudaStream_t st) {
    if (s.head_dim == 128) return launch_kh<2>(s, sp, a, st, false, 0, 1.0);
    if (s.head_dim == 64) return launch_kh<1>(s, sp, a, st, false, 0, 1.0);
    set_error("kvc_score: tensor-core path needs head_dim 64 or 128");
    return KVC_ERR_UNSUPPORTED;
}

int launch_score_tc_keyformer(const kvc_shape &s, const ScoreSplit &sp, const ScoreArgs &a,
                              uint64_t seed, double tau, cudaStream_t st) {
    if (s.head_dim == 128) return launch_kh<2>(s, sp, a, st, true, seed, tau);
    if (s.head_dim == 64) return launch_kh<1>(s, sp, a, st, true, seed, tau);
    set_error("kvc_score_keyformer: tensor-core path needs head_dim 64 or 128");
    return KVC_ERR_UNSUPPORTED;
}

}  // namespace kvc
