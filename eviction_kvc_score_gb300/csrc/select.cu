// select.cu -- ZigZagKV MBA, layer budgets and per-head top-K.
//
// MBA (blog post "ZigZagKV, KVCache 80% compression near-lossless", section
// "ZigZagKV's new observations"): the fewest tokens whose scores reach 90%
// of a head's attention mass.  Mass is exact fixed point u = floor(c*2^56),
// so the count does not depend on summation order.  Instead of sorting, an
// MSB radix select over the fp32 bit patterns (non-negative floats order like
// their bit patterns) keeps, per digit bucket, the count and the u-mass, and
// descends into the bucket where the running mass from the top first reaches
// the threshold.  The exact crossing value v* and the mass above it then give
// the count in closed form.
//
// Budgets (same post, "ZigZagKV space allocation"): integer proportional
// split with a floor and largest remainders, capped at the prefix length.
//
// Top-K (same post, "SnapKV" / "ZigZagKV token selection"): radix select of
// the B-th largest prefix score, then an ordered block-wide compaction that
// keeps everything above it and the lowest-index ties, writing positions in
// ascending order.
//
// Histograms: one shared histogram per block with a 12-bit first digit
// (exponent plus four mantissa bits, so a head's scores spread over many
// buckets).  Within a warp the lanes that share the first active lane's digit
// are added as one group (ballot + warp reductions), the rest one by one.
// Only native 32-bit shared atomics are used: the exact 64-bit mass of a
// bucket is a (hi, lo) word pair, lo's carry folded into hi.
#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kBuckets = 4096;
constexpr int kPasses = 3;

// A valid score is a non-negative float, so its sign bit is zero and its
// 31-bit pattern orders like its value.  Three radix digits, most significant
// first: bits 30..19 (exponent and top mantissa bits), 18..9, 8..0.
__device__ __forceinline__ int digit_shift(int pass) { return pass == 0 ? 19 : pass == 1 ? 9 : 0; }
__device__ __forceinline__ int digit_bits(int pass) { return pass == 0 ? 12 : pass == 1 ? 10 : 9; }

__device__ __forceinline__ int digit_of(uint32_t key, int pass) {
    return (int)((key >> digit_shift(pass)) & ((1u << digit_bits(pass)) - 1u));
}

// Does key lie inside the bucket chosen by the earlier passes?
__device__ __forceinline__ bool in_prefix(uint32_t key, int pass, uint32_t prefix) {
    return pass == 0 || (key >> digit_shift(pass - 1)) == prefix;
}

// floor(c * 2^56) for a float 0 <= c <= 1, from its bits with integer
// operations only (exact): c = m * 2^(e-150) with the 24-bit significand m,
// so c * 2^56 = m * 2^(e-94).
__device__ __forceinline__ unsigned long long fixed56(uint32_t key) {
    const int e = (int)(key >> 23);
    if (e == 0) return 0;   // zero and subnormals: below 2^-126
    const unsigned long long m = (key & 0x7FFFFFu) | 0x800000u;
    const int sh = e - 94;
    if (sh >= 0) return m << sh;   // sh <= 33 for c <= 1
    if (sh <= -24) return 0;
    return m >> (-sh);
}

// Called by all 32 lanes of one warp.  Walks the nb buckets from the largest
// digit down and finds the first one at which the running total (base plus
// everything above) reaches the target, as decided by reach(total).  Lane L
// owns the buckets [nb-(L+1)per, nb-L*per); the lanes scan their range sums
// and the first lane whose range reaches walks its own buckets.  That lane
// stores the bucket, the total strictly above it and the count strictly above
// it to *chosen, *above, *cabove (shared memory).
template <typename V, typename VA, typename Reach>
__device__ __forceinline__ void find_bucket(const VA *val, const uint32_t *cnt, int nb, V base,
                                            long long cbase, Reach reach, int *chosen, V *above,
                                            long long *cabove) {
    const int lane = threadIdx.x & 31;
    const int per = nb / 32;
    const int lo = nb - (lane + 1) * per;
    V ls = 0;
    long long lc = 0;
    for (int k = 0; k < per; ++k) {   // staggered order: no bank conflicts
        const int d = lo + ((k + lane) & (per - 1));
        ls += (V)val[d];
        lc += cnt[d];
    }
    V incl = ls;
    long long incl_c = lc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const V a = __shfl_up_sync(0xffffffffu, incl, o);
        const long long b = __shfl_up_sync(0xffffffffu, incl_c, o);
        if (lane >= o) {
            incl += a;
            incl_c += b;
        }
    }
    const unsigned mask = __ballot_sync(0xffffffffu, reach(base + incl));
    const int finder = mask ? __ffs(mask) - 1 : 31;   // no lane: corrupt input
    if (lane == finder) {
        V run = base + incl - ls;
        long long runc = cbase + incl_c - lc;
        int pick = lo;
        for (int d = lo + per - 1; d >= lo; --d) {
            if (reach(run + (V)val[d])) {
                pick = d;
                break;
            }
            run += (V)val[d];
            runc += cnt[d];
        }
        *chosen = pick;
        *above = run;
        *cabove = runc;
    }
}

// ------------------------------------------------------------------ MBA
struct MbaSmem {
    uint32_t cnt[kBuckets];
    uint32_t lo[kBuckets];
    uint32_t hi[kBuckets];
    unsigned long long msum[kBuckets];
};

__device__ __forceinline__ void add_mass(MbaSmem &sm, int d, unsigned long long x) {
    const uint32_t lo = (uint32_t)x;
    const uint32_t old = atomicAdd(&sm.lo[d], lo);
    atomicAdd(&sm.hi[d], (uint32_t)(x >> 32) + (old + lo < old ? 1u : 0u));
}

__global__ void __launch_bounds__(kSelThreads)
    mba_kernel(const float *__restrict__ scores, int T, uint32_t num, uint32_t den,
               int32_t *__restrict__ mba, uint32_t *status) {
    extern __shared__ __align__(16) uint8_t sel_smem[];
    MbaSmem &sm = *reinterpret_cast<MbaSmem *>(sel_smem);
    __shared__ unsigned long long s_total, s_sum_gt;
    __shared__ long long s_cnt_gt;
    __shared__ uint32_t s_prefix;
    __shared__ int s_bad, s_done, s_chosen;
    const float *c = scores + (int64_t)blockIdx.x * T;
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        s_sum_gt = 0;
        s_cnt_gt = 0;
        s_prefix = 0;
        s_bad = 0;
        s_done = 0;
    }
    for (int pass = 0; pass < kPasses; ++pass) {
        const int nb = 1 << digit_bits(pass);
        for (int i = tid; i < nb; i += kSelThreads) {
            sm.cnt[i] = 0;
            sm.lo[i] = 0;
            sm.hi[i] = 0;
        }
        __syncthreads();
        const uint32_t prefix = s_prefix;
        const int lane = tid & 31;
        for (int base = 0; base < T; base += kSelThreads) {   // uniform trip count
            const int j = base + tid;
            const float v = j < T ? c[j] : 0.f;
            const uint32_t key = __float_as_uint(v);
            if (pass == 0 && j < T && !(v >= 0.f && v <= 1.f)) s_bad = 1;
            const bool valid = j < T && key <= 0x3F800000u && in_prefix(key, pass, prefix);
            const unsigned vmask = __ballot_sync(0xffffffffu, valid);
            if (vmask == 0) continue;
            // peel the first valid lane's digit: its lanes add as one group
            const int d = digit_of(key, pass);
            const int leader = __ffs(vmask) - 1;
            const int dl = __shfl_sync(0xffffffffu, d, leader);
            const bool same = valid && d == dl;
            const unsigned smask = __ballot_sync(0xffffffffu, same);
            const unsigned long long u = valid ? fixed56(key) : 0ull;
            const unsigned long long us = same ? u : 0ull;
            const unsigned s0 = __reduce_add_sync(0xffffffffu, (unsigned)(us & 0x7FFFu));
            const unsigned s1 = __reduce_add_sync(0xffffffffu, (unsigned)((us >> 15) & 0x7FFFu));
            const unsigned s2 = __reduce_add_sync(0xffffffffu, (unsigned)((us >> 30) & 0x7FFFu));
            const unsigned s3 = __reduce_add_sync(0xffffffffu, (unsigned)(us >> 45));
            if (lane == leader) {
                atomicAdd(&sm.cnt[dl], (uint32_t)__popc(smask));
                add_mass(sm, dl, (unsigned long long)s0 + ((unsigned long long)s1 << 15) +
                                     ((unsigned long long)s2 << 30) + ((unsigned long long)s3 << 45));
            }
            if (valid && !same) {
                atomicAdd(&sm.cnt[d], 1u);
                add_mass(sm, d, u);
            }
        }
        __syncthreads();
        for (int d = tid; d < nb; d += kSelThreads)
            sm.msum[d] = ((unsigned long long)sm.hi[d] << 32) + sm.lo[d];
        __syncthreads();
        if (warp == 0) {
            if (pass == 0) {
                unsigned long long tot = 0;
                for (int d = tid; d < nb; d += 32) tot += sm.msum[d];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
                if (tid == 0) {
                    s_total = tot;
                    // a head whose scores sum above 16 (or hold invalid values)
                    // would overflow the exact comparisons below
                    if (s_bad || tot > (1ull << 60)) s_bad = 1;
                    if (s_bad || (unsigned __int128)num * tot == 0) s_done = 1;
                }
                __syncwarp();
            }
            if (!s_done) {
                const unsigned __int128 need = (unsigned __int128)num * s_total;
                find_bucket<unsigned long long>(
                    sm.msum, sm.cnt, nb, s_sum_gt, s_cnt_gt,
                    [&](unsigned long long x) { return (unsigned __int128)den * x >= need; },
                    &s_chosen, &s_sum_gt, &s_cnt_gt);
                __syncwarp();
                if (tid == 0) s_prefix = (prefix << digit_bits(pass)) | (uint32_t)s_chosen;
            }
        }
        __syncthreads();
        if (s_done) break;
    }
    if (tid == 0) {
        if (s_bad) {
            set_status(status, KVC_DEV_BAD_SCORE);
            mba[blockIdx.x] = 0;
        } else if (s_done) {
            mba[blockIdx.x] = 0;
        } else {
            // s_prefix is now the exact crossing value v*; every element above
            // it is counted in s_cnt_gt / s_sum_gt; ties at v* each carry u*.
            const unsigned long long ustar = fixed56(s_prefix);
            const unsigned __int128 need = (unsigned __int128)num * s_total;
            const unsigned __int128 have = (unsigned __int128)den * s_sum_gt;
            const unsigned __int128 step = (unsigned __int128)den * ustar;
            if (step == 0 || have >= need) {
                // unreachable for valid scores (the crossing bucket always
                // carries mass); never divide by zero on corrupt input
                set_status(status, KVC_DEV_BAD_SCORE);
                mba[blockIdx.x] = (int32_t)s_cnt_gt;
            } else {
                const long long k = (long long)((need - have + step - 1) / step);
                mba[blockIdx.x] = (int32_t)(s_cnt_gt + k);
            }
        }
    }
}

// ------------------------------------------------------------------ budgets
// One block, one thread per layer (L <= 1024).  Integer arithmetic only.
constexpr int kMaxLayers = 1024;

// floor(a*b/c) and the remainder, exact (64-bit when the product fits).
__device__ __forceinline__ void muldiv(unsigned long long a, unsigned long long b,
                                       unsigned long long c, unsigned long long &q,
                                       unsigned long long &r) {
    if (b == 0 || a <= ~0ull / b) {
        const unsigned long long p = a * b;
        q = p / c;
        r = p % c;
    } else {
        const unsigned __int128 p = (unsigned __int128)a * b;
        q = (unsigned long long)(p / c);
        r = (unsigned long long)(p % c);
    }
}

// Largest-remainder split of R over the eligible layers by weight S (equal
// weights if the eligible weights sum to 0): every layer gets
// floor(R S_l / sum S); the leftover units go one each to the largest
// remainders, ties to the lower layer.  Returns the calling thread's share.
__device__ long long lr_split(int L, const long long *S, const unsigned char *elig, long long R,
                              long long *rem, unsigned long long *red) {
    const int l = threadIdx.x;
    const bool act = l < L;
    if (l == 0) red[0] = red[1] = red[2] = 0;
    __syncthreads();
    const bool e = act && elig[l];
    if (e) {
        atomicAdd(&red[0], (unsigned long long)S[l]);
        atomicAdd(&red[1], 1ull);
    }
    __syncthreads();
    unsigned long long sumw = red[0];
    const unsigned long long n_el = red[1];
    if (n_el == 0 || R <= 0) {
        __syncthreads();
        return 0;
    }
    const bool equal = sumw == 0;
    if (equal) sumw = n_el;
    long long add = 0;
    if (e) {
        unsigned long long q, r;
        muldiv((unsigned long long)R, equal ? 1ull : (unsigned long long)S[l], sumw, q, r);
        add = (long long)q;
        rem[l] = (long long)r;
        atomicAdd(&red[2], q);
    }
    __syncthreads();
    const long long left = R - (long long)red[2];
    if (e && left > 0) {
        long long rank = 0;
        for (int o = 0; o < L; ++o)
            rank += elig[o] && (rem[o] > rem[l] || (rem[o] == rem[l] && o < l));
        if (rank < left) add += 1;
    }
    __syncthreads();
    return add;
}

__global__ void __launch_bounds__(kMaxLayers)
    budget_kernel(const int32_t *__restrict__ mba, int L, int Hkv, long long P, long long total,
                  long long floor_, int32_t *__restrict__ budget) {
    __shared__ long long S[kMaxLayers], rem[kMaxLayers];
    __shared__ unsigned char elig[kMaxLayers];
    __shared__ unsigned long long red[3];
    const int l = threadIdx.x;
    const bool act = l < L;
    if (total >= (long long)L * P) {
        if (act) budget[l] = (int32_t)P;
        return;
    }
    if (act) {
        long long acc = 0;
        for (int k = 0; k < Hkv; ++k) acc += mba[(int64_t)l * Hkv + k];
        S[l] = acc;
        elig[l] = 1;
    }
    __syncthreads();
    long long B = floor_ + lr_split(L, S, elig, total - (long long)L * floor_, rem, red);
    while (true) {
        if (l == 0) red[0] = 0;
        __syncthreads();
        if (act && B > P) {
            atomicAdd(&red[0], (unsigned long long)(B - P));
            B = P;
        }
        __syncthreads();
        const unsigned long long excess = red[0];
        __syncthreads();
        if (excess == 0) break;
        if (act) elig[l] = B < P;
        __syncthreads();
        B += lr_split(L, S, elig, (long long)excess, rem, red);
    }
    if (act) budget[l] = (int32_t)B;
}

// Per-head budgets: block l splits the layer's H_kv * B_l tokens over its
// heads by MBA (the same largest-remainder split, no per-head minimum), caps
// each head at P and re-splits the excess over the uncapped heads.  One
// thread per head (H_kv <= 1024).
__global__ void __launch_bounds__(kMaxLayers)
    head_budget_kernel(const int32_t *__restrict__ mba, const int32_t *__restrict__ budget, int Hkv,
                       long long P, int32_t *__restrict__ head_budget) {
    __shared__ long long S[kMaxLayers], rem[kMaxLayers];
    __shared__ unsigned char elig[kMaxLayers];
    __shared__ unsigned long long red[3];
    const int l = blockIdx.x, k = threadIdx.x;
    const bool act = k < Hkv;
    long long Bl = budget[l];
    Bl = Bl < 0 ? 0 : (Bl > P ? P : Bl);
    if (act) {
        S[k] = mba[(int64_t)l * Hkv + k];
        elig[k] = 1;
    }
    __syncthreads();
    long long B = lr_split(Hkv, S, elig, (long long)Hkv * Bl, rem, red);
    while (true) {
        if (k == 0) red[0] = 0;
        __syncthreads();
        if (act && B > P) {
            atomicAdd(&red[0], (unsigned long long)(B - P));
            B = P;
        }
        __syncthreads();
        const unsigned long long excess = red[0];
        __syncthreads();
        if (excess == 0) break;
        if (act) elig[k] = B < P;
        __syncthreads();
        B += lr_split(Hkv, S, elig, (long long)excess, rem, red);
    }
    if (act) head_budget[(int64_t)l * Hkv + k] = (int32_t)B;
}

// ------------------------------------------------------------------ top-K
// Block-wide exclusive scan of one uint32 per thread.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *warp_tot, uint32_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t a = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += a;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t w = lane < kSelWarps ? warp_tot[lane] : 0u;
        uint32_t wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t a = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += a;
        }
        if (lane < kSelWarps) warp_tot[lane] = wi - w;   // exclusive
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    const uint32_t r = warp_tot[warp] + incl - v;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kSelThreads)
    topk_kernel(const float *__restrict__ scores, int T, int P, int Hkv,
                const int32_t *__restrict__ budget, int per_head, int k_max,
                int32_t *__restrict__ idx, uint32_t *status) {
    __shared__ uint32_t cnt[kBuckets];
    __shared__ uint32_t warp_tot[32];
    __shared__ uint32_t s_total;
    __shared__ uint32_t s_prefix;
    __shared__ long long s_cnt_gt, s_dummy;
    __shared__ int s_bad, s_chosen;
    const int head = blockIdx.x;
    const int l = head / Hkv;
    const int tid = threadIdx.x, warp = tid >> 5;
    const float *c = scores + (int64_t)head * T;
    int32_t *out = idx + (int64_t)head * k_max;
    long long B = per_head ? budget[head] : budget[l];
    if (B < 0) {
        if (tid == 0) set_status(status, KVC_DEV_BAD_BUDGET);
        B = 0;
    }
    if (B > P) B = P;
    if (B > k_max) {
        if (tid == 0) set_status(status, KVC_DEV_BAD_BUDGET);
        B = k_max;
    }
    if (B == 0) return;
    if (B == P) {
        for (int j = tid; j < P; j += kSelThreads) out[j] = j;
        return;
    }
    if (tid == 0) {
        s_prefix = 0;
        s_cnt_gt = 0;
        s_bad = 0;
    }
    for (int pass = 0; pass < kPasses; ++pass) {
        const int nb = 1 << digit_bits(pass);
        for (int i = tid; i < nb; i += kSelThreads) cnt[i] = 0;
        __syncthreads();
        const uint32_t prefix = s_prefix;
        const int lane = tid & 31;
        for (int base = 0; base < P; base += kSelThreads) {
            const int j = base + tid;
            const float v = j < P ? c[j] : 0.f;
            const uint32_t key = __float_as_uint(v);
            if (pass == 0 && j < P && !(v >= 0.f)) s_bad = 1;
            const bool valid = j < P && in_prefix(key, pass, prefix);
            const unsigned vmask = __ballot_sync(0xffffffffu, valid);
            if (vmask == 0) continue;
            const int d = digit_of(key, pass);
            const int leader = __ffs(vmask) - 1;
            const int dl = __shfl_sync(0xffffffffu, d, leader);
            const bool same = valid && d == dl;
            const unsigned smask = __ballot_sync(0xffffffffu, same);
            if (lane == leader) atomicAdd(&cnt[dl], (uint32_t)__popc(smask));
            if (valid && !same) atomicAdd(&cnt[d], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            // counts stand in for the values: walk until B elements are reached
            find_bucket<long long>(
                cnt, cnt, nb, s_cnt_gt, 0, [&](long long x) { return x >= B; }, &s_chosen,
                &s_cnt_gt, &s_dummy);
            __syncwarp();
            if (tid == 0) s_prefix = (prefix << digit_bits(pass)) | (uint32_t)s_chosen;
        }
        __syncthreads();
    }
    if (tid == 0 && s_bad) set_status(status, KVC_DEV_BAD_SCORE);
    const uint32_t vstar = s_prefix;
    const long long need_eq = B - s_cnt_gt;   // >= 1
    // Ordered compaction: position of a kept j is G(j) + min(E(j), need_eq)
    // with G/E the numbers of elements above / equal to v* before j.
    long long g_before = 0, e_before = 0;
    for (int base = 0; base < P; base += 4 * kSelThreads) {
        const int j0 = base + 4 * tid;
        uint32_t gt[4], eq[4];
        uint32_t ng = 0, ne = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = j0 + i;
            const uint32_t key = j < P ? __float_as_uint(c[j]) : 0u;
            gt[i] = (j < P) && key > vstar;
            eq[i] = (j < P) && key == vstar;
            ng += gt[i];
            ne += eq[i];
        }
        const uint32_t packed = block_excl_scan(ng | (ne << 16), warp_tot, &s_total);
        long long G = g_before + (packed & 0xFFFFu);
        long long E = e_before + (packed >> 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (gt[i] || (eq[i] && E < need_eq)) {
                const long long pos = G + (E < need_eq ? E : need_eq);
                if (pos < B) out[pos] = j0 + i;   // always true for valid scores
            }
            G += gt[i];
            E += eq[i];
        }
        const uint32_t tot = s_total;
        g_before += tot & 0xFFFFu;
        e_before += tot >> 16;
        if (g_before + (e_before < need_eq ? e_before : need_eq) >= B) break;
        __syncthreads();
    }
}

// Threshold selection: per head, every prefix position with score >= tau,
// ascending (ordered block compaction), at most k_max written; counts[head]
// is the full number (more than k_max sets KVC_DEV_BAD_BUDGET).
__global__ void __launch_bounds__(kSelThreads)
    threshold_kernel(const float *__restrict__ scores, int T, int P, float tau, int k_max,
                     int32_t *__restrict__ idx, int32_t *__restrict__ counts, uint32_t *status) {
    __shared__ uint32_t warp_tot[32];
    __shared__ uint32_t s_total;
    const int head = blockIdx.x;
    const int tid = threadIdx.x;
    const float *c = scores + (int64_t)head * T;
    int32_t *out = idx + (int64_t)head * k_max;
    long long before = 0;
    for (int base = 0; base < P; base += 4 * kSelThreads) {
        const int j0 = base + 4 * tid;
        uint32_t keep[4], nk = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = j0 + i;
            keep[i] = (j < P) && c[j] >= tau;
            nk += keep[i];
        }
        long long pos = before + block_excl_scan(nk, warp_tot, &s_total);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (keep[i]) {
                if (pos < k_max) out[pos] = j0 + i;
                ++pos;
            }
        }
        before += s_total;
        __syncthreads();
    }
    if (tid == 0) {
        counts[head] = (int32_t)min(before, (long long)INT32_MAX);
        if (before > k_max) set_status(status, KVC_DEV_BAD_BUDGET);
    }
}

}  // namespace

int launch_head_budget(const kvc_shape &s, const int32_t *mba, const int32_t *budget,
                       int32_t *head_budget, cudaStream_t st) {
    if (s.n_kv_heads > kMaxLayers) {
        set_error("kvc_head_budget: at most %d KV heads", kMaxLayers);
        return KVC_ERR_UNSUPPORTED;
    }
    head_budget_kernel<<<s.n_layers, (s.n_kv_heads + 31) / 32 * 32, 0, st>>>(
        mba, budget, s.n_kv_heads, (long long)s.seq_len - s.window, head_budget);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_head_budget: launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

int launch_threshold(const kvc_shape &s, const float *scores, float tau, int32_t k_max,
                     int32_t *idx, int32_t *counts, uint32_t *status, cudaStream_t st) {
    const int heads = s.n_layers * s.n_kv_heads;
    threshold_kernel<<<heads, kSelThreads, 0, st>>>(scores, s.seq_len, s.seq_len - s.window, tau,
                                                    k_max, idx, counts, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_threshold_select: launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

int launch_mba(const kvc_shape &s, const float *scores, uint32_t num, uint32_t den, int32_t *mba,
               uint32_t *status, cudaStream_t st) {
    const int heads = s.n_layers * s.n_kv_heads;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(mba_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(MbaSmem));
        attr = true;
    }
    mba_kernel<<<heads, kSelThreads, sizeof(MbaSmem), st>>>(scores, s.seq_len, num, den, mba, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_mba_budget: MBA launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

int launch_budget(const kvc_shape &s, const int32_t *mba, int64_t total, int32_t floor_,
                  int32_t *budget, cudaStream_t st) {
    if (s.n_layers > kMaxLayers) {
        set_error("kvc_mba_budget: at most %d layers", kMaxLayers);
        return KVC_ERR_UNSUPPORTED;
    }
    budget_kernel<<<1, (s.n_layers + 31) / 32 * 32, 0, st>>>(mba, s.n_layers, s.n_kv_heads,
                                    (long long)s.seq_len - s.window, (long long)total,
                                    (long long)floor_, budget);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_mba_budget: budget launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

int launch_topk(const kvc_shape &s, const float *scores, const int32_t *budget, int per_head,
                int32_t k_max, int32_t *idx, uint32_t *status, cudaStream_t st) {
    const int heads = s.n_layers * s.n_kv_heads;
    topk_kernel<<<heads, kSelThreads, 0, st>>>(scores, s.seq_len, s.seq_len - s.window,
                                                s.n_kv_heads, budget, per_head, k_max, idx, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_topk_select: launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

}  // namespace kvc
