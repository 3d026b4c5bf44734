// select.cu -- ZigZagKV MBA, layer budgets and per-head top-K (and the
// optional per-head budgets and threshold selection).
//
// MBA (blog post "ZigZagKV, KVCache 80% compression near-lossless", section
// "ZigZagKV's new observations"): the fewest tokens whose scores reach 90%
// of a head's attention mass.  Mass is exact fixed point u = floor(c*2^56),
// so the count does not depend on summation order.  Instead of sorting, an
// MSB radix select over the fp32 bit patterns (non-negative floats order like
// their bit patterns) finds the crossing value v* -- the score at which the
// running mass from the top first reaches the threshold -- and the exact
// mass above it gives the count in closed form.  The first digit's bucket is
// found from truncated bucket masses and confirmed with one exact pass; the two
// remaining digits use exact 64-bit bucket masses.
//
// Budgets (same post, "ZigZagKV space allocation"): integer proportional
// split with a floor and largest remainders, capped at the prefix length.
//
// Top-K (same post, "SnapKV" / "ZigZagKV token selection"): radix select of
// the B-th largest prefix score, then an ordered block-wide compaction that
// keeps everything above it and the lowest-index ties, writing positions in
// ascending order.
//
// One 1024-thread block per head; the head's scores are read from global
// memory once and kept in shared memory for the later passes (when they fit,
// T <= 36,864); every bucket search is a block-wide scan with one to four
// buckets per thread.  Only native 32-bit shared atomics are used: a 64-bit
// bucket mass is a (hi, lo) word pair, lo's carry folded into hi.
#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
// ------------------------------------------------------------------ scans
// Block-wide exclusive scan of one value per thread (1024 threads); *total
// receives the block sum.  warp_tot must hold 32 values.
template <typename V>
__device__ __forceinline__ V block_scan_excl(V v, V *warp_tot, V *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    V incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const V a = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += a;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const V w = warp_tot[lane];
        V wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const V a = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += a;
        }
        warp_tot[lane] = wi - w;
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    const V r = warp_tot[warp] + incl - v;
    __syncthreads();
    return r;
}

// Block sum; total must point to shared memory (the scan's last lane writes
// it, every thread reads it after the scan's barriers).
template <typename V>
__device__ __forceinline__ V block_sum(V v, V *warp_tot, V *total) {
    (void)block_scan_excl(v, warp_tot, total);
    return *total;
}

// floor(c * 2^56) for 0 <= c <= 1, from the bits: a normal c is
// m 2^(e - 150) with m its 24-bit significand, so the floor is m shifted by
// e - 94 (left, or right with the dropped bits truncated); a subnormal c is
// below 2^-126 and its floor is 0 (the shift right by 94 gives that).
// Integer shifts instead of a float-to-64-bit conversion per score: the
// conversion shares the SM's special-function pipe and cost ~13% of the MBA
// kernel.
__device__ __forceinline__ unsigned long long fixed56f(float c) {
    const uint32_t bits = __float_as_uint(c);
    const int e = (int)(bits >> 23);
    const unsigned long long m = (bits & 0x7FFFFFu) | (e ? 0x800000u : 0u);
    const int sh = e - 94;
    return sh >= 0 ? (m << sh) : (sh > -64 ? (m >> -sh) : 0ull);
}

// floor(c * 2^27) for 0 <= c <= 1 the same way (shift e - 123); 2^27 at c = 1.
__device__ __forceinline__ uint32_t fixed27f(float c) {
    const uint32_t bits = __float_as_uint(c);
    const int e = (int)(bits >> 23);
    const uint32_t m = (bits & 0x7FFFFFu) | (e ? 0x800000u : 0u);
    const int sh = e - 123;
    return sh >= 0 ? (m << sh) : (sh > -32 ? (m >> -sh) : 0u);
}

// Copy n floats of one head from global to shared memory with many loads in
// flight per thread (16-byte vectors when the row is 16-byte aligned), so
// the later passes never wait on global-memory latency.
__device__ __forceinline__ void stage_scores(const float *__restrict__ g, float *sm, int n) {
    const int tid = threadIdx.x;
    if ((reinterpret_cast<uintptr_t>(g) & 15) == 0) {
        const int n4 = n >> 2;
        const float4 *g4 = reinterpret_cast<const float4 *>(g);
        float4 *s4 = reinterpret_cast<float4 *>(sm);
        for (int base = 0; base < n4; base += 8 * kSelThreads) {
            float4 r[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = base + i * kSelThreads + tid;
                if (k < n4) r[i] = g4[k];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = base + i * kSelThreads + tid;
                if (k < n4) s4[k] = r[i];
            }
        }
        for (int j = (n4 << 2) + tid; j < n; j += kSelThreads) sm[j] = g[j];
    } else {
        for (int base = 0; base < n; base += 8 * kSelThreads) {
            float r[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = base + i * kSelThreads + tid;
                if (k < n) r[i] = g[k];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = base + i * kSelThreads + tid;
                if (k < n) sm[k] = r[i];
            }
        }
    }
}

// Visit scores 0..n-1 of one head: thread tid gets k = base + i*1024 + tid,
// sixteen loads issued before any is used (latency hidden when the scores come
// from global memory).  f(k, v, in) is called for every lane, with in false
// past the end, so warp-wide votes inside f stay uniform.
template <typename F>
__device__ __forceinline__ void for_scores(const float *__restrict__ src, int n, F f) {
    constexpr int kBatch = 16;
    const int tid = threadIdx.x;
    for (int base = 0; base < n; base += kBatch * kSelThreads) {
        float r[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int k = base + i * kSelThreads + tid;
            r[i] = k < n ? src[k] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int k = base + i * kSelThreads + tid;
            f(k, r[i], k < n);
        }
    }
}

// ------------------------------------------------------------------ MBA
// Per head (one 1024-thread block): the scores are read once from global
// memory into shared memory (when they fit), then
//  1. a 4096-bucket histogram of the top 12 key bits with counts and
//     truncated 32-bit masses (native shared atomics), and the exact total
//     U = sum u_j in per-thread 64-bit sums;
//  2. the truncated masses point to the bucket d1 where the running mass
//     from the top reaches num/den of the total; one exact pass (64-bit per-thread
//     sums) checks it -- den * A < num * U <= den * (A + M_d1), A the exact
//     mass above d1 -- and steps to the neighbouring non-empty bucket in the
//     rare case rounding picked the wrong one;
//  3. two exact radix passes (10 and 9 bits, 64-bit masses as (hi, lo) word
//     pairs) inside that bucket find the crossing value v*;
// each bucket search is a block-wide scan, one bucket per thread.  The count
// then follows in closed form from the exact mass above v*.
constexpr int kCacheFloats = 36864;   // scores per head kept in shared memory (144 KiB)
constexpr int kB0 = 4096;

__device__ __forceinline__ void add_mass64(uint32_t *lo, uint32_t *hi, int d, unsigned long long x) {
    const uint32_t l = (uint32_t)x;
    const uint32_t old = atomicAdd(&lo[d], l);
    atomicAdd(&hi[d], (uint32_t)(x >> 32) + (old + l < old ? 1u : 0u));
}

__global__ void __launch_bounds__(kSelThreads)
    mba_kernel(const float *__restrict__ scores, int T, uint32_t num, uint32_t den, int cached,
               int32_t *__restrict__ mba, uint32_t *status) {
    extern __shared__ __align__(16) uint8_t sel_smem[];
    uint32_t *cnt = reinterpret_cast<uint32_t *>(sel_smem);   // [4096]
    uint32_t *fm = cnt + kB0;                                   // [4096] floor(c * 2^27) sums
    uint32_t *lo = fm + kB0;                                    // [1024]
    uint32_t *hi = lo + 1024;                                   // [1024]
    float *cache = reinterpret_cast<float *>(hi + 1024);        // [T] when cached
    __shared__ unsigned long long wt64[32], s_tot64;
    __shared__ uint32_t wt32[32], s_tot32;
    __shared__ int s_d, s_step;
    __shared__ unsigned long long s_add;
    __shared__ long long s_cadd;
    const int tid = threadIdx.x;
    const float *c = scores + (int64_t)blockIdx.x * T;
    const float *src = cached ? cache : c;

    // 1. histogram, exact total
    for (int i = tid; i < kB0; i += kSelThreads) {
        cnt[i] = 0;
        fm[i] = 0u;
    }
    if (cached) stage_scores(c, cache, T);
    __syncthreads();
    unsigned long long my_u = 0;
    int bad = 0;
    for_scores(src, T, [&](int, float v, bool in) {
        const bool valid = in && v >= 0.f && v <= 1.f;
        if (in && !valid) bad = 1;
        if (!valid) return;
        const int d = (int)(__float_as_uint(v) >> 19);
        my_u += fixed56f(v);
        atomicAdd(&cnt[d], 1u);
        atomicAdd(&fm[d], fixed27f(v));   // guide mass, truncated
    });
    bad = __syncthreads_or(bad);
    const unsigned long long U = block_sum(my_u, wt64, &s_tot64);
    if (bad || U > (1ull << 60)) {   // invalid scores, or a head summing above 16
        if (tid == 0) {
            set_status(status, KVC_DEV_BAD_SCORE);
            mba[blockIdx.x] = 0;
        }
        return;
    }
    if (U == 0 || num == 0) {
        if (tid == 0) mba[blockIdx.x] = 0;
        return;
    }
    const unsigned __int128 need = (unsigned __int128)num * U;

    // 2. guide from the truncated masses (floor(c 2^27) per element, at most
    // T units below the exact mass): thread t holds buckets 4095-4t ..
    // 4092-4t (descending)
    uint32_t f4[4], fl = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f4[i] = fm[kB0 - 1 - 4 * tid - i];
        fl += f4[i];
    }
    const uint32_t fpre = block_scan_excl(fl, wt32, &s_tot32);
    const unsigned long long target = ((unsigned long long)s_tot32 * num + den - 1) / den;
    if (tid == 0) s_d = -1;
    __syncthreads();
    {
        unsigned long long run = fpre;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (f4[i] > 0 && run < target && run + f4[i] >= target)
                atomicMax(&s_d, kB0 - 1 - 4 * tid - i);
            run += f4[i];
        }
    }
    __syncthreads();
    if (tid == 0 && s_d < 0) {   // rounding left the target unreached: lowest non-empty bucket
        int d = 0;
        while (d < kB0 - 1 && cnt[d] == 0) ++d;
        s_d = d;
    }
    __syncthreads();
    // exact check of the bucket, moving one non-empty bucket at a time
    unsigned long long A = 0;
    long long C = 0;
    for (int iter = 0; iter < kB0; ++iter) {
        const int d1 = s_d;
        unsigned long long a = 0, m = 0;
        uint32_t cg = 0;
        for_scores(src, T, [&](int, float v, bool in) {
            const int d = (int)(__float_as_uint(v) >> 19);
            const unsigned long long u = in ? fixed56f(v) : 0ull;
            if (d > d1) {
                a += u;
                cg += in;
            } else if (d == d1) {
                m += u;
            }
        });
        A = block_sum(a, wt64, &s_tot64);
        const unsigned long long M = block_sum(m, wt64, &s_tot64);
        C = (long long)block_sum(cg, wt32, &s_tot32);
        if (tid == 0) {
            s_step = 0;
            if ((unsigned __int128)den * A >= need) {
                int d = d1 + 1;
                while (d < kB0 - 1 && cnt[d] == 0) ++d;
                s_d = d;
                s_step = 1;
            } else if ((unsigned __int128)den * (A + M) < need) {
                int d = d1 - 1;
                while (d > 0 && cnt[d] == 0) --d;
                s_d = d;
                s_step = 1;
            }
        }
        __syncthreads();
        if (!s_step) break;
    }
    // 3. exact radix passes inside the bucket
    uint32_t prefix = (uint32_t)s_d;
    for (int pass = 1; pass < 3; ++pass) {
        const int bits = pass == 1 ? 10 : 9, shift = pass == 1 ? 9 : 0, nb = 1 << bits;
        for (int i = tid; i < nb; i += kSelThreads) {
            cnt[i] = 0;
            lo[i] = 0;
            hi[i] = 0;
        }
        __syncthreads();
        for_scores(src, T, [&](int, float v, bool in) {
            const uint32_t key = __float_as_uint(v);
            if (!in || (key >> (shift + bits)) != prefix) return;
            const int dd = (int)((key >> shift) & (uint32_t)(nb - 1));
            atomicAdd(&cnt[dd], 1u);
            add_mass64(lo, hi, dd, fixed56f(v));
        });
        __syncthreads();
        // thread t holds bucket nb-1-t (descending); threads past nb hold 0
        const int b = nb - 1 - tid;
        const unsigned long long mb = b >= 0 ? ((unsigned long long)hi[b] << 32) | lo[b] : 0ull;
        const uint32_t cb = b >= 0 ? cnt[b] : 0u;
        const unsigned long long mpre = block_scan_excl(mb, wt64, &s_tot64);
        const uint32_t cpre = block_scan_excl(cb, wt32, &s_tot32);
        if (mb > 0 && (unsigned __int128)den * (A + mpre) < need &&
            (unsigned __int128)den * (A + mpre + mb) >= need) {
            s_d = b;
            s_add = mpre;
            s_cadd = cpre;
        }
        __syncthreads();
        A += s_add;
        C += s_cadd;
        prefix = (prefix << bits) | (uint32_t)s_d;
        __syncthreads();
    }
    if (tid == 0) {
        // prefix is the crossing value v*; the elements above it carry A and
        // number C; each tie at v* adds u*
        const unsigned long long ustar = fixed56f(__uint_as_float(prefix));
        const unsigned __int128 have = (unsigned __int128)den * A;
        const unsigned __int128 step = (unsigned __int128)den * ustar;
        long long m;
        if (step == 0 || have >= need) {
            set_status(status, KVC_DEV_BAD_SCORE);   // unreachable for valid scores
            m = C;
        } else {
            m = C + (long long)((need - have + step - 1) / step);
        }
        if (kDebugBounds && (m < 0 || m > T)) set_status(status, KVC_DEV_INVARIANT);
        mba[blockIdx.x] = (int32_t)m;
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
                  long long floor_, int32_t *__restrict__ budget, uint32_t *status) {
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
    if (kDebugBounds) {   // sum = total (every layer at P if total >= L P), floor <= B <= P
        __syncthreads();
        if (l == 0) red[0] = 0;
        __syncthreads();
        if (act) {
            atomicAdd(&red[0], (unsigned long long)B);
            if (B < floor_ || B > P) set_status(status, KVC_DEV_INVARIANT);
        }
        __syncthreads();
        if (l == 0 && (long long)red[0] != total) set_status(status, KVC_DEV_INVARIANT);
    }
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
                const int32_t *__restrict__ budget, int per_head, int k_max, int cached,
                int32_t *__restrict__ idx, uint32_t *status) {
    extern __shared__ __align__(16) uint8_t sel_smem[];
    uint32_t *cnt = reinterpret_cast<uint32_t *>(sel_smem);   // [4096]
    float *cache = reinterpret_cast<float *>(cnt + kB0);        // [P] when cached
    __shared__ uint32_t warp_tot[32];
    __shared__ uint32_t s_total;
    __shared__ int s_d;
    __shared__ uint32_t s_cadd;
    const int head = blockIdx.x;
    const int l = head / Hkv;
    const int tid = threadIdx.x;
    const float *c = scores + (int64_t)head * T;
    const float *src = cached ? cache : c;
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
    // radix select of the B-th largest key: 12 bits (4096 buckets), then 10
    // and 9 bits inside the chosen bucket; each bucket search is a block-wide
    // scan, one or four buckets per thread
    for (int i = tid; i < kB0; i += kSelThreads) cnt[i] = 0;
    if (cached) stage_scores(c, cache, P);
    __syncthreads();
    int bad = 0;
    for_scores(src, P, [&](int, float v, bool in) {
        if (!in) return;
        if (!(v >= 0.f)) bad = 1;
        atomicAdd(&cnt[(__float_as_uint(v) >> 19) & (kB0 - 1)], 1u);
    });
    bad = __syncthreads_or(bad);
    if (tid == 0 && bad) set_status(status, KVC_DEV_BAD_SCORE);
    // B is clamped to [0, P] above and P < 2^31: positions and counts from
    // here on are 32-bit (64-bit integer arithmetic cost ~8% of the kernel)
    int C = 0;   // elements strictly above the current bucket
    {
        uint32_t c4[4], cl = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            c4[i] = cnt[kB0 - 1 - 4 * tid - i];
            cl += c4[i];
        }
        uint32_t run = block_scan_excl(cl, warp_tot, &s_total);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (c4[i] > 0 && run < B && run + c4[i] >= B) {
                s_d = kB0 - 1 - 4 * tid - i;
                s_cadd = run;
            }
            run += c4[i];
        }
        __syncthreads();
        C = s_cadd;
    }
    uint32_t prefix = (uint32_t)s_d;
    for (int pass = 1; pass < 3; ++pass) {
        const int bits = pass == 1 ? 10 : 9, shift = pass == 1 ? 9 : 0, nb = 1 << bits;
        __syncthreads();
        for (int i = tid; i < nb; i += kSelThreads) cnt[i] = 0;
        __syncthreads();
        for_scores(src, P, [&](int, float v, bool in) {
            const uint32_t key = __float_as_uint(v);
            if (in && (key >> (shift + bits)) == prefix)
                atomicAdd(&cnt[(key >> shift) & (uint32_t)(nb - 1)], 1u);
        });
        __syncthreads();
        const int b = nb - 1 - tid;
        const uint32_t cb = b >= 0 ? cnt[b] : 0u;
        const uint32_t cpre = block_scan_excl(cb, warp_tot, &s_total);
        if (cb > 0 && C + cpre < B && C + cpre + cb >= B) {
            s_d = b;
            s_cadd = cpre;
        }
        __syncthreads();
        C += s_cadd;
        prefix = (prefix << bits) | (uint32_t)s_d;
    }
    const uint32_t vstar = prefix;
    const int need_eq = (int)B - C;   // >= 1
    // Ordered compaction: position of a kept j is G(j) + min(E(j), need_eq)
    // with G/E the numbers of elements above / equal to v* before j.
    int g_before = 0, e_before = 0;
    uint32_t nxt[4];   // next chunk's keys, loaded before this chunk's scan
#pragma unroll
    for (int i = 0; i < 4; ++i) nxt[i] = 4 * tid + i < P ? __float_as_uint(src[4 * tid + i]) : 0u;
    for (int base = 0; base < P; base += 4 * kSelThreads) {
        const int j0 = base + 4 * tid;
        uint32_t gt[4], eq[4];
        uint32_t ng = 0, ne = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = j0 + i;
            const uint32_t key = nxt[i];
            gt[i] = (j < P) && key > vstar;
            eq[i] = (j < P) && key == vstar;
            ng += gt[i];
            ne += eq[i];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int jn = j0 + 4 * kSelThreads + i;
            nxt[i] = jn < P ? __float_as_uint(src[jn]) : 0u;
        }
        const uint32_t packed = block_excl_scan(ng | (ne << 16), warp_tot, &s_total);
        int G = g_before + (int)(packed & 0xFFFFu);
        int E = e_before + (int)(packed >> 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (gt[i] || (eq[i] && E < need_eq)) {
                const int pos = G + (E < need_eq ? E : need_eq);
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
    if (kDebugBounds) {   // B positions, strictly ascending, inside the prefix
        __syncthreads();
        for (int i = tid; i < B; i += kSelThreads) {
            const int32_t x = out[i];
            if (x < 0 || x >= P || (i > 0 && out[i - 1] >= x)) set_status(status, KVC_DEV_INVARIANT);
        }
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
    if (kDebugBounds) {   // written positions strictly ascending, inside the prefix
        __syncthreads();
        const long long n = before < k_max ? before : k_max;
        for (long long i = tid; i < n; i += kSelThreads) {
            const int32_t x = out[i];
            if (x < 0 || x >= P || (i > 0 && out[i - 1] >= x)) set_status(status, KVC_DEV_INVARIANT);
        }
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
    const int cached = s.seq_len <= kCacheFloats;
    const size_t smem = (size_t)(2 * kB0 + 2 * 1024) * 4 + (cached ? (size_t)s.seq_len * 4 : 0);
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(mba_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (2 * kB0 + 2 * 1024 + kCacheFloats) * 4);
        attr = true;
    }
    mba_kernel<<<heads, kSelThreads, smem, st>>>(scores, s.seq_len, num, den, cached, mba, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_mba_budget: MBA launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

int launch_budget(const kvc_shape &s, const int32_t *mba, int64_t total, int32_t floor_,
                  int32_t *budget, uint32_t *status, cudaStream_t st) {
    if (s.n_layers > kMaxLayers) {
        set_error("kvc_mba_budget: at most %d layers", kMaxLayers);
        return KVC_ERR_UNSUPPORTED;
    }
    budget_kernel<<<1, (s.n_layers + 31) / 32 * 32, 0, st>>>(mba, s.n_layers, s.n_kv_heads,
                                    (long long)s.seq_len - s.window, (long long)total,
                                    (long long)floor_, budget, status);
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
    const int P = s.seq_len - s.window;
    const int cached = P <= kCacheFloats;
    const size_t smem = (size_t)kB0 * 4 + (cached ? (size_t)P * 4 : 0);
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (kB0 + kCacheFloats) * 4);
        attr = true;
    }
    topk_kernel<<<heads, kSelThreads, smem, st>>>(scores, s.seq_len, P, s.n_kv_heads, budget,
                                                   per_head, k_max, cached, idx, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_topk_select: launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

}  // namespace kvc
