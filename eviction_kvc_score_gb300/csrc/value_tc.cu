// value_tc.cu -- THINKV value-channel scores on the sm_103a tensor cores.
//
// What is computed ("ThinK: Thinner Key Cache by Query-Driven Pruning",
// appendix "Value cache pruning strategy"): for every unit = (layer, KV head)
// and window row r (position P + w, w = r mod W) the attention output
//   o_r = sum over keys j <= P + w of 2^(x_rj + nb_r) v_j,
//   x_rj = q_r . k_j log2(e) / sqrt(D),  nb_r = -(m_r + log2 l_r)
// (nb_r from the score pass's pass 1 + merge, so each probability is final
// when formed), and score_v[d] = sum_r o_r[d]^2 over the unit's G*W rows.
//
// Work item = (unit, job): a job is 256 of the unit's window rows, the full
// M of one SM-pair MMA.  Items are dealt round-robin to the pairs, so with two
// jobs per unit and an even number of pairs, pairs 2m and 2m+1 run the two
// jobs of the same unit side by side and the second reader of each K/V tile
// finds it in L2.  Per 128-key tile of an item:
//   MMA1  S = Q K^T           M = 256 rows, N = 128 keys, K = D = 128
//         (A = the CTA's 128 Q rows, B = the CTA's 64 keys, both K-major,
//          128-byte swizzled as TMA writes them) -> a TMEM slot
//   epi   p = 2^(s log2(e)/sqrt(D) + nb_r), 0 where row r does not see key j,
//         split into bf16 p_hi = p truncated to its top 16 bits and p_lo =
//         bf16(p - p_hi) (about 16 significant bits together) and stored back
//         into the slot (tcgen05.st)
//   MMA2  O += P_hi V + P_lo V   M = 256 rows, N = 128 channels, K = 128 keys
//         (A = P straight from TMEM, B = the CTA's 64 channels of the tile's
//          128 value rows, channel-contiguous: the MN-major B layout)
// A single bf16 P (8 bits) moved the squared norms of a head with few window
// rows by up to 3e-3; the two-term split brings every score within 1e-4 of
// the fp64 definition at the price of a second P V product.
// O accumulates in TMEM over chunks of kChunkTiles tiles, each chunk added
// into fp32 sums in shared memory by the epilogue; at the item's end each
// epilogue thread squares its row's 32 channels and a warp butterfly sums them
// over the warp's 32 rows, giving one partial per (unit, job, CTA, warp) --
// reduced in a fixed order afterwards, so the result is deterministic.
//
// TMEM (512 columns per CTA): O in columns [0,128); three S/P slots of 128
// columns at 128, 256, 384.  Within a slot, epilogue warpgroup e reads S
// columns [32e, 32e+32) (keys 32e..) in two halves of 16 and writes each
// half's 8 P_hi and 8 P_lo words back into its own 16 columns (one MMA K-step
// of P: hi words, then lo words), so no thread overwrites S that it or
// another thread has not yet read; it also owns O channels [32e, 32e+32).
//
// Roles per CTA: warp 0 loads Q rows (per item) and K (per tile, its 64
// keys) into a three-stage K ring; warp 19 loads V (its 64 channels of the
// tile's 128 keys) into a three-stage V ring; warp 1 issues S = Q K^T (even
// CTA) or relays Q/K load completions to the even CTA (odd CTA); warp 18
// issues O += P V (even CTA) or relays V completions (odd CTA); warps 2..17
// are four epilogue warpgroups (four warps per SM sub-partition hide the
// exponentials' latency; two left the kernel at 40% of its MMA time).
// Two issuing threads because one thread's issue loop, not the tensor
// pipe, set the pace: measured on the 32K prompt, a single issuer spent
// ~2,300 clocks per tile issuing its 24 MMAs (1,536 clocks of tensor time);
// split, `kvc_channel_prune_value` went from 3.84 to 3.20 ms with identical
// scores.  K and V have rings of their own, K freed as soon as a tile's S is
// computed (a shared stage freed only after the tile's P V left the S issuer
// idle ~1,200 clocks per tile waiting for K): 3.13 ms; the rings' free
// signals folded into the slot barriers: 3.06 ms.  Per accumulator the MMAs
// keep their order, so the result does not depend on the split.  Every wait is bounded
// (kvc_internal.cuh).
#include "kvc_internal.cuh"

namespace kvc {

namespace {

// K and V rings of as many stages as there are S/P slots and indexed like
// them, so a slot's barriers also free its stages: K stage s when the slot's
// S is computed (s_full), V stage s when its P V is done (slot_empty) -- one
// commit per issuer and tile fewer than rings of their own.
constexpr int kKStages = 3;
constexpr int kVvStages = 3;
constexpr int kVSlots = 3;
constexpr int kVTileKeys = 128;                 // keys per pair tile
// O is accumulated in TMEM over chunks of this many tiles (2048 keys, 256
// MMAs) and each chunk is added into fp32 registers by the epilogue: the
// tensor core's fp32 accumulation loses about half an ulp per MMA in one
// direction, which over a 32K-key item (4096 MMAs) moved O by ~2.5e-4.
constexpr int kChunkTiles = 16;
constexpr int kVEWG = 4;                        // epilogue warpgroups
constexpr int kVKeysWG = kVTileKeys / kVEWG;    // S columns (keys) and O channels per warpgroup
constexpr int kVThreadsTC = 64 + 128 * kVEWG + 64;   // + the P V issuer and V loader warps
constexpr int kPVWarp = 2 + 4 * kVEWG;                // P V issuer (even CTA) / V relay (odd)
constexpr int kVLoadWarp = kPVWarp + 1;               // V loader
constexpr uint32_t kVTmemCols = 512;
constexpr uint32_t kOCol = 0;                   // O accumulator columns [0,128)
constexpr uint32_t kSlotCol0 = 128;             // slot s at 128 + 128 s
constexpr int kQBox = 128 * 128;                // 128 rows x 64 bf16
constexpr int kKBox = 64 * 128;                 // 64 keys x 64 bf16
constexpr int kVBox = 128 * 128;                // 128 keys x 64 channels
constexpr int kKStageBytes = 2 * kKBox;          // head_dim 128: two K boxes
constexpr int kVStageBytes = kVBox;

struct VtcParams {
    int64_t n_units;
    int njob;             // jobs (256-row blocks) per unit
    int64_t n_items;      // n_units * njob
    int pairs;
    int T, P, W, rows, rows_pad, n_tiles;
    float cs;             // log2(e) / sqrt(D)
    const float *neg_bias;
    float *partial;       // [units][kValueTcParts = (job, CTA, warp)][128]
    uint32_t *status;
};

struct VSmem {
    uint8_t *q;        // [2][128 rows][128 B]
    uint8_t *k;        // [kKStages][K box 0 | K box 1]
    uint8_t *v;        // [kVvStages][V box]
    float *oacc;       // [16 epilogue warps][32 channels][32 lanes]: O summed over chunks
    uint64_t *kf, *kp;   // K ring [kKStages]: loaded, peer's loaded (even CTA)
    uint64_t *vf, *vp;   // V ring [kVvStages]
    uint64_t *q_full, *q_empty, *q_pfull;
    uint64_t *s_full, *p_full, *slot_empty;   // [slots]
    uint64_t *o_full, *o_empty, *drain, *drain2;
    uint32_t *tmem_base;
    volatile int *abort_flag;
};

constexpr size_t kOaccBytes = (size_t)4 * kVEWG * kVKeysWG * 32 * sizeof(float);
constexpr size_t kVSmemBytes = 1024 + 2 * kQBox + (size_t)kKStages * kKStageBytes +
                               (size_t)kVvStages * kVStageBytes + kOaccBytes +
                               (2 * kKStages + 2 * kVvStages + 3 * kVSlots + 9) * 8 +
                               16;

__device__ __forceinline__ VSmem vcarve(uint8_t *raw) {
    VSmem s;
    uint8_t *b = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.q = b;
    b += 2 * kQBox;
    s.k = b;
    b += (size_t)kKStages * kKStageBytes;
    s.v = b;
    b += (size_t)kVvStages * kVStageBytes;
    s.oacc = reinterpret_cast<float *>(b);
    b += kOaccBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(b);
    s.kf = bars;
    s.kp = bars + kKStages;
    s.vf = bars + 2 * kKStages;
    s.vp = s.vf + kVvStages;
    s.q_full = s.vf + 2 * kVvStages;
    s.q_empty = s.q_full + 1;
    s.q_pfull = s.q_full + 2;
    s.s_full = s.q_full + 3;
    s.p_full = s.s_full + kVSlots;
    s.slot_empty = s.p_full + kVSlots;
    s.o_full = s.slot_empty + kVSlots;
    s.o_empty = s.o_full + 1;
    s.drain = s.o_full + 2;
    s.drain2 = s.o_full + 3;
    s.tmem_base = reinterpret_cast<uint32_t *>(s.drain2 + 1);
    s.abort_flag = reinterpret_cast<volatile int *>(s.tmem_base + 1);
    return s;
}

// Items of pair c: c, c + pairs, c + 2 pairs, ...
struct Item {
    int64_t u;
    int job;
};
__device__ __forceinline__ Item item_of(int64_t i, int njob) {
    Item it;
    it.u = i / njob;
    it.job = (int)(i % njob);
    return it;
}

// K-major 128-byte swizzled operand (8-row groups 1024 bytes apart), as TMA
// writes a box whose inner extent is 128 bytes.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(lbo >> 4) << 16;
    d |= static_cast<uint64_t>(sbo >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(96)
    value_out_tc(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, VtcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const VSmem s = vcarve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)cluster_ctarank();
    const int64_t c = cluster_id_x();
    if (threadIdx.x == 0) {
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(&s.kf[i], 1);
            mbar_init(&s.kp[i], 1);
        }
        for (int i = 0; i < kVvStages; ++i) {
            mbar_init(&s.vf[i], 1);
            mbar_init(&s.vp[i], 1);
        }
        mbar_init(s.q_full, 1);
        mbar_init(s.q_empty, 1);
        mbar_init(s.q_pfull, 1);
        for (int i = 0; i < kVSlots; ++i) {
            mbar_init(&s.s_full[i], 1);
            mbar_init(&s.p_full[i], 2 * 4 * kVEWG);   // every epilogue warp of both CTAs
            mbar_init(&s.slot_empty[i], 1);
        }
        mbar_init(s.o_full, 1);
        mbar_init(s.o_empty, 2 * 4 * kVEWG);
        mbar_init(s.drain, 1);
        mbar_init(s.drain2, 1);
        *s.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc2(s.tmem_base, kVTmemCols);
        tmem_relinquish2();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *s.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            uint32_t gt = 0, qi = 0;
            uint32_t issued = 0;
            bool ok = true;
            for (int64_t i = c; i < p.n_items && ok; i += p.pairs) {
                const Item it = item_of(i, p.njob);
                if (qi > 0 && !mbar_wait(s.q_empty, (qi - 1) & 1, s.abort_flag, p.status)) break;
                mbar_arrive_expect_tx(s.q_full, 2u * kQBox);
                for (int kh = 0; kh < 2; ++kh)
                    tma_load_3d(&tq, s.q_full, s.q + kh * kQBox, kh * 64, it.job * 256 + rank * 128,
                                (int)it.u);
                ++qi;
                for (int t = 0; t < p.n_tiles; ++t, ++gt) {
                    const uint32_t st = gt % kKStages, ph = (gt / kKStages) & 1;
                    // stage st is free once the slot-st S of three tiles ago is
                    // computed (its s_full phase); the first round needs no wait
                    if (gt >= (uint32_t)kKStages &&
                        !mbar_wait(&s.s_full[st], ph ^ 1, s.abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t *stage = s.k + (size_t)st * kKStageBytes;
                    mbar_arrive_expect_tx(&s.kf[st], (uint32_t)kKStageBytes);
                    for (int kh = 0; kh < 2; ++kh)
                        tma_load_3d(&tk, &s.kf[st], stage + kh * kKBox, kh * 64,
                                    t * kVTileKeys + rank * 64, (int)it.u);
                    ++issued;
                }
            }
            if (*s.abort_flag) {   // unwind: every copy started must land
                for (uint32_t g = issued > kKStages ? issued - kKStages : 0; g < issued; ++g)
                    mbar_drain(&s.kf[g % kKStages], (g / kKStages) & 1);
                if (qi > 0) mbar_drain(s.q_full, (qi - 1) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 1) {
            // ------------------------------------------------ relay (odd CTA)
            const uint32_t r_pfull = mapa_shared(smem_u32(s.kp), 0);
            const uint32_t r_qpfull = mapa_shared(smem_u32(s.q_pfull), 0);
            uint32_t gt = 0, qi = 0;
            bool ok = true;
            for (int64_t i = c; i < p.n_items && ok; i += p.pairs) {
                if (!mbar_wait(s.q_full, qi & 1, s.abort_flag, p.status)) break;
                mbar_arrive_remote(r_qpfull);
                ++qi;
                for (int t = 0; t < p.n_tiles; ++t, ++gt) {
                    const uint32_t st = gt % kKStages, ph = (gt / kKStages) & 1;
                    if (!mbar_wait(&s.kf[st], ph, s.abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_remote(r_pfull + st * 8u);
                }
            }
        } else if (lane == 0) {
            // ------------------------------------------------ S = Q K^T issuer (even CTA)
            constexpr uint16_t kBoth = 3;
            const uint32_t idesc1 = idesc_bf16_f32(256, 128);   // both K-major
            uint32_t gt = 0, qi = 0;
            bool ok = true;
            const uint64_t qd0 = desc_sw128(smem_u32(s.q), 16u, 1024u);
            for (int64_t i = c; i < p.n_items && ok; i += p.pairs) {
                if (!mbar_wait(s.q_full, qi & 1, s.abort_flag, p.status)) break;
                if (!mbar_wait(s.q_pfull, qi & 1, s.abort_flag, p.status)) break;
                ++qi;
                for (int t = 0; t < p.n_tiles; ++t, ++gt) {
                    const uint32_t st = gt % kKStages, ph = (gt / kKStages) & 1;
                    const uint32_t slot = gt % kVSlots, use = gt / kVSlots;
                    if (!mbar_wait(&s.kf[st], ph, s.abort_flag, p.status) ||
                        !mbar_wait(&s.kp[st], ph, s.abort_flag, p.status) ||
                        !mbar_wait(&s.slot_empty[slot], (use & 1) ^ 1, s.abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t kd0 = desc_sw128(smem_u32(s.k + (size_t)st * kKStageBytes), 16u, 1024u);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        // K-steps 0-3 in the first 64-column box, 4-7 in the
                        // second; 32 bytes each
                        const int kh = ks >> 2, off = (ks & 3) * 32;
                        const uint64_t a = qd0 + (uint64_t)((kh * kQBox + off) >> 4);
                        const uint64_t b = kd0 + (uint64_t)((kh * kKBox + off) >> 4);
                        tc_mma2_bf16(tmem + kSlotCol0 + slot * 128, a, b, idesc1, ks > 0);
                    }
                    tc_commit2(&s.s_full[slot], kBoth);
                    if (t == p.n_tiles - 1) tc_commit2(s.q_empty, kBoth);
                }
            }
            tc_commit2(s.drain, 1);
            mbar_drain(s.drain, 0);
        }
    } else if (warp == kPVWarp) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------ O += P V issuer (even CTA)
            // The second issuing thread.
            constexpr uint16_t kBoth = 3;
            const uint32_t idesc2 = idesc_bf16_f32(256, 128) | (1u << 16);  // B MN-major
            uint32_t gt = 0, chunks = 0;
            bool ok = true;
            for (int64_t i = c; i < p.n_items && ok; i += p.pairs) {
                for (int t = 0; t < p.n_tiles; ++t, ++gt) {
                    const uint32_t slot = gt % kVSlots, use = gt / kVSlots;
                    const uint32_t st = gt % kVvStages, ph = (gt / kVvStages) & 1;
                    const bool first = t % kChunkTiles == 0;
                    const bool last = t % kChunkTiles == kChunkTiles - 1 || t == p.n_tiles - 1;
                    if (!mbar_wait(&s.vf[st], ph, s.abort_flag, p.status) ||
                        !mbar_wait(&s.vp[st], ph, s.abort_flag, p.status) ||
                        !mbar_wait(&s.p_full[slot], use & 1, s.abort_flag, p.status) ||
                        (first && !mbar_wait(s.o_empty, (chunks & 1) ^ 1, s.abort_flag, p.status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t scol = tmem + kSlotCol0 + slot * 128;
                    const uint64_t b0 = desc_sw128(smem_u32(s.v + (size_t)st * kVStageBytes), 1024u, 1024u);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        // keys 16 ks ..: the P_hi words of that half of warpgroup
                        // ks / 2's keys at columns 16 ks, its P_lo words 8
                        // further; value rows 16 ks .. of the box (2048 bytes on)
                        const uint32_t acol = scol + (uint32_t)(ks * 16);
                        const uint64_t b = b0 + (uint64_t)(ks * (2048 >> 4));
                        tc_mma2_bf16_tmem_a(tmem + kOCol, acol, b, idesc2, (first && ks == 0) ? 0u : 1u);
                        tc_mma2_bf16_tmem_a(tmem + kOCol, acol + 8u, b, idesc2, 1u);
                    }
                    tc_commit2(&s.slot_empty[slot], kBoth);
                    if (last) {
                        tc_commit2(s.o_full, kBoth);
                        ++chunks;
                    }
                }
            }
            tc_commit2(s.drain2, 1);
            mbar_drain(s.drain2, 0);
        } else if (lane == 0) {
            // ------------------------------------------------ V relay (odd CTA)
            const uint32_t r_vp = mapa_shared(smem_u32(s.vp), 0);
            uint32_t gt = 0;
            bool ok = true;
            for (int64_t i = c; i < p.n_items && ok; i += p.pairs) {
                for (int t = 0; t < p.n_tiles; ++t, ++gt) {
                    const uint32_t st = gt % kVvStages, ph = (gt / kVvStages) & 1;
                    if (!mbar_wait(&s.vf[st], ph, s.abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_remote(r_vp + st * 8u);
                }
            }
        }
    } else if (warp == kVLoadWarp) {
        if (lane == 0) {
            // ------------------------------------------------ V loader
            tma_prefetch_desc(&tv);
            uint32_t gt = 0, issued = 0;
            bool ok = true;
            for (int64_t i = c; i < p.n_items && ok; i += p.pairs) {
                const Item it = item_of(i, p.njob);
                for (int t = 0; t < p.n_tiles; ++t, ++gt) {
                    const uint32_t st = gt % kVvStages, ph = (gt / kVvStages) & 1;
                    // free once the slot-st P V of three tiles ago is done
                    if (!mbar_wait(&s.slot_empty[st], ph ^ 1, s.abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&s.vf[st], (uint32_t)kVStageBytes);
                    tma_load_3d(&tv, &s.vf[st], s.v + (size_t)st * kVStageBytes, rank * 64,
                                t * kVTileKeys, (int)it.u);
                    ++issued;
                }
            }
            if (*s.abort_flag) {   // unwind: every copy started must land
                for (uint32_t g = issued > kVvStages ? issued - kVvStages : 0; g < issued; ++g)
                    mbar_drain(&s.vf[g % kVvStages], (g / kVvStages) & 1);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const int ewg = (warp - 2) >> 2;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t r_pfull = mapa_shared(smem_u32(s.p_full), 0);
        const uint32_t r_oempty = mapa_shared(smem_u32(s.o_empty), 0);
        uint32_t gt = 0, chunks = 0;
        bool ok = true;
        for (int64_t i = c; i < p.n_items && ok; i += p.pairs) {
            const Item it = item_of(i, p.njob);
            const int r = it.job * 256 + rank * 128 + quarter * 32 + lane;
            const bool real = r < p.rows;
            const float nb = real ? p.neg_bias[it.u * p.rows_pad + r] : -INFINITY;
            const int lim_row = p.P + (real ? r % p.W : 0);   // last key the row sees
            // this row's O, channels [32 ewg, +32), summed over chunks in
            // shared memory (registers stay free for a whole tile of S)
            float *acc = s.oacc + (size_t)(warp - 2) * kVKeysWG * 32 + lane;
#pragma unroll
            for (int k = 0; k < kVKeysWG; ++k) acc[k * 32] = 0.f;
            for (int t = 0; t < p.n_tiles; ++t, ++gt) {
                const uint32_t slot = gt % kVSlots, use = gt / kVSlots;
                if (!mbar_wait(&s.s_full[slot], use & 1, s.abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // this warpgroup's 32 keys, read at once; each half of 16 (one
                // MMA K-step) gets its P words (8 hi, then 8 lo) written back
                // into its own 16 S columns, both halves in one store
                const uint32_t scol = tmem + lane_base + kSlotCol0 + slot * 128 + ewg * kVKeysWG;
                float v[32];
                tmem_ld32(scol, v);
                tmem_ld_wait();
                reg_fence(v);
                const int lim = lim_row - (t * kVTileKeys + ewg * kVKeysWG);
                if (lim < kVKeysWG - 1) {   // the window's causal edge: mask invisible keys
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i > lim) v[i] = -INFINITY;   // 2^-inf = +0
                }
                const unsigned long long cs2 = f2_pack(p.cs, p.cs), nb2 = f2_pack(nb, nb);
                uint32_t w[32];
#pragma unroll
                for (int i2 = 0; i2 < 16; ++i2) {
                    float y0, y1;
                    f2_unpack(f2_fma(f2_pack(v[2 * i2], v[2 * i2 + 1]), cs2, nb2), y0, y1);
                    const float p0 = ex2(y0), p1 = ex2(y1);
                    // p = hi + lo: hi keeps the top 16 bits (truncated, a
                    // bf16), lo = p - hi is exact and rounded to bf16
                    const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
                    const unsigned long long lo2 = f2_add(
                        f2_pack(p0, p1), f2_pack(-__uint_as_float(b0 & 0xFFFF0000u),
                                                 -__uint_as_float(b1 & 0xFFFF0000u)));
                    float l0, l1;
                    f2_unpack(lo2, l0, l1);
                    uint32_t hi, lo;
                    // lower 16 bits: the even key (first along K)
                    asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(hi) : "r"(b0), "r"(b1));
                    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(l1), "f"(l0));
                    // half i2 / 8: hi words at 16 half + i2 % 8, lo words 8 further
                    w[(i2 >> 3) * 16 + (i2 & 7)] = hi;
                    w[(i2 >> 3) * 16 + 8 + (i2 & 7)] = lo;
                }
                tmem_st32(scol, w);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                // the stores are complete (wait::st) and fenced for the
                // thread sync: hand the slot to the MMA issuer
                if (lane == 0) mbar_arrive_remote(r_pfull + slot * 8u);
                if (t % kChunkTiles == kChunkTiles - 1 || t == p.n_tiles - 1) {
                    // a chunk of O is complete: add it to the registers
                    if (!mbar_wait(s.o_full, chunks & 1, s.abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    ++chunks;
                    tc_fence_after();
                    const uint32_t ocol = tmem + lane_base + kOCol + ewg * kVKeysWG;
                    {
                        float o[32];
                        tmem_ld32(ocol, o);
                        tmem_ld_wait();
                        reg_fence(o);
#pragma unroll
                        for (int k = 0; k < 32; ++k) acc[k * 32] += o[k];
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote(r_oempty);   // O may be overwritten
                }
            }
            if (!ok) break;
            // squares summed over the warp's 32 rows: a butterfly that halves
            // the vector each step leaves lane l with channel l
            float a[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) a[k] = acc[k * 32] * acc[k * 32];
#pragma unroll
            for (int half = 16; half >= 1; half >>= 1) {
                const bool upper = (lane & half) != 0;   // lane bit that chooses the kept half
#pragma unroll
                for (int k = 0; k < half; ++k) {
                    const float send = upper ? a[k] : a[k + half];
                    const float keep = upper ? a[k + half] : a[k];
                    a[k] = keep + __shfl_xor_sync(0xffffffffu, send, half);
                }
            }
            // one partial per (job, CTA, warp): no barrier between warps, so
            // a warp that gave up on a wait cannot leave another one waiting
            p.partial[(it.u * kValueTcParts + (it.job * 2 + rank) * 4 + quarter) * 128 +
                      ewg * kVKeysWG + lane] = a[0];
        }
    }
    // teardown: no MMA, load or remote arrive of the pair is left
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc2(tmem, kVTmemCols);
    }
    cluster_sync_all();
}

}  // namespace

bool value_tc_eligible(const kvc_shape &s) {
    const int G = s.n_q_heads / s.n_kv_heads;
    return s.dtype == KVC_BF16 && s.head_dim == 128 && (int64_t)G * s.window <= kMaxRowsTC;
}

int launch_value_tc(const kvc_shape &s, const ScoreSplit &sp, const void *q, const void *k,
                    const void *v, const float *neg_bias, float *partial, uint32_t *status,
                    cudaStream_t st, int *parts_out) {
    if (!value_tc_eligible(s) || sp.rows_pad % 256 || sp.rows_pad > kMaxRowsTC) {
        set_error("kvc_channel_prune_value: tensor-core kernel needs bf16, head_dim 128 and "
                  "G*W <= 512 with the tensor-core row split");
        return KVC_ERR_UNSUPPORTED;
    }
    const int G = s.n_q_heads / s.n_kv_heads;
    CUtensorMap tq, tk, tv;
    const uint64_t units = (uint64_t)sp.n_units;
    if (!make_tma_map(&tq, q, 128, (uint64_t)G * s.window, units, 128) ||
        !make_tma_map(&tk, k, 128, (uint64_t)s.seq_len, units, 64) ||
        !make_tma_map(&tv, v, 128, (uint64_t)s.seq_len, units, 128)) {
        set_error("kvc_channel_prune_value: cuTensorMapEncodeTiled failed (alignment or driver)");
        return KVC_ERR_CUDA;
    }
    VtcParams p;
    p.n_units = sp.n_units;
    p.njob = sp.rows_pad / 256;
    p.n_items = sp.n_units * p.njob;
    const int pairs = score_tc_pairs(0);
    p.pairs = (int)(p.n_items < pairs ? p.n_items : pairs);
    p.T = s.seq_len;
    p.P = s.seq_len - s.window;
    p.W = s.window;
    p.rows = sp.rows;
    p.rows_pad = sp.rows_pad;
    p.n_tiles = (s.seq_len + kVTileKeys - 1) / kVTileKeys;
    p.cs = (float)(kLog2e / sqrt(128.0));
    p.neg_bias = neg_bias;
    p.partial = partial;
    p.status = status;
    cudaFuncSetAttribute(value_out_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)kVSmemBytes);
    value_out_tc<<<2 * p.pairs, kVThreadsTC, kVSmemBytes, st>>>(tq, tk, tv, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_channel_prune_value: tensor-core launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    *parts_out = 8 * p.njob;   // the first 8 njob of the kValueTcParts slots
    return KVC_OK;
}

}  // namespace kvc
