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
// mass above it gives the count in closed form.  Every bucket of the first
// digit holds scores of one float exponent, which makes its exact mass a sum
// of 24-bit integers shifted by a per-bucket amount: one pass gives exact
// bucket masses with 32-bit shared atomics.
//
// Budgets (same post, "ZigZagKV space allocation"): integer proportional
// split with a floor and largest remainders, capped at the prefix length.
//
// Top-K (same post, "SnapKV" / "ZigZagKV token selection"): radix select of
// the B-th largest prefix score, then an ordered block-wide compaction that
// keeps everything above it and the lowest-index ties, writing positions in
// ascending order.
//
// One block per head: 1024 threads, or for MBA 512 threads two per SM when
// the heads exceed one wave of 1024-thread blocks.  The first pass copies the
// head's scores into shared memory (cp.async, when they fit) for the later
// passes; a second pass gathers the crossing bucket's keys into per-warp
// shared lists, so that the two remaining digits never reread the row (for
// top-K on a held row that pass is also the compaction's classification).
// The last MBA block to finish computes the layer budgets.  Bucket searches
// are block-wide scans with one to eight buckets per thread; only native
// 32-bit shared atomics are used on the usual path (64-bit shared atomics are
// emulated and several times slower).
#include "kvc_internal.cuh"

#include <mutex>

namespace kvc {

namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
// ------------------------------------------------------------------ scans
template <typename V>
__device__ __forceinline__ V shfl_up(V v, int o) {
    return __shfl_up_sync(0xffffffffu, v, o);
}
__device__ __forceinline__ unsigned __int128 shfl_up(unsigned __int128 v, int o) {
    const unsigned long long lo = __shfl_up_sync(0xffffffffu, (unsigned long long)v, o);
    const unsigned long long hi = __shfl_up_sync(0xffffffffu, (unsigned long long)(v >> 64), o);
    return ((unsigned __int128)hi << 64) | lo;
}

// Block-wide exclusive scan of one value per thread (a block of any multiple
// of 32 threads up to 1024); *total receives the block sum.  warp_tot must
// hold 32 values.
template <typename V>
__device__ __forceinline__ V block_scan_excl(V v, V *warp_tot, V *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    V incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const V a = shfl_up(incl, o);
        if (lane >= o) incl += a;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = (int)(blockDim.x >> 5);
        const V w = lane < nw ? warp_tot[lane] : V{};
        V wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const V a = shfl_up(wi, o);
            if (lane >= o) wi += a;
        }
        if (lane < nw) warp_tot[lane] = wi - w;
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

// Order key of a score: its bit pattern without the sign bit.  Non-negative
// floats order like their bit patterns, and -0.0 becomes +0.0 (the two
// compare equal); a negative score, already reported as invalid, takes its
// magnitude's key in every pass alike, and no key's bucket leaves [0, 4096).
__device__ __forceinline__ uint32_t skey(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }

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

// Visit scores 0..n-1 of one head (NT-thread block): thread tid gets
// k = base + i*NT + tid,
// sixteen loads issued before any is used (latency hidden when the scores come
// from global memory).  f(k, v, in) is called for every lane, with in false
// past the end, so warp-wide votes inside f stay uniform.
template <int NT = kSelThreads, typename F>
__device__ __forceinline__ void for_scores(const float *__restrict__ src, int n, F f) {
    constexpr int kBatch = 16;
    const int tid = threadIdx.x;
    for (int base = 0; base < n; base += kBatch * NT) {
        float r[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int k = base + i * NT + tid;
            r[i] = k < n ? src[k] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int k = base + i * NT + tid;
            f(k, r[i], k < n);
        }
    }
}

// ------------------------------------------------------------------ MBA
// Per head (one block of NT threads):
//  1. one pass over the scores (copying them into shared memory when they
//     fit, for the later passes) builds a 4096-bucket histogram of the top 12
//     key bits holding each bucket's EXACT mass: every score of a bucket has
//     the same float exponent e, so u = floor(c * 2^56) is w * 2^s with
//     s = max(e - 94, 0) and w < 2^24 an integer (the significand, or the
//     floor itself for tiny c); the bucket sums w (two 32-bit shared atomics
//     of its 12-bit halves, or one 64-bit atomic for rows above 2^20 scores)
//     and its mass is that sum shifted by s;
//  2. one block-wide 128-bit scan of the masses from the top gives the total
//     U (exact at any size, so a head summing above 16 is caught) and the
//     bucket d1 where the running mass first reaches num/den of U;
//  3. one more pass counts the scores above d1 and gathers d1's keys into
//     per-warp shared lists;
//  4. the two remaining digits (10 and 9 bits) are histogrammed from the
//     lists alone;
// each digit's bucket is found by one scan of packed (count, mass) pairs; the
// count then follows in closed form from the exact mass above the crossing
// value v*.
constexpr int kCacheFloats = 36864;   // scores per head kept in shared memory (144 KiB)
constexpr int kB0 = 4096;
// Above this many scores a bucket's 32-bit halves could overflow; longer rows
// accumulate w with one 64-bit atomic instead (emulated, several times slower).
constexpr int kSplitMaxT = 1 << 20;
// Smallest gather list a block is launched with.
constexpr int kMinList = 1024;

using u128 = unsigned __int128;

// w for key bits of a score in [0, 1]: floor(c * 2^56) >> max(e - 94, 0).
__device__ __forceinline__ uint32_t unit_mass(uint32_t key) {
    const uint32_t e = key >> 23;
    const uint32_t m = (key & 0x7FFFFFu) | (e ? 0x800000u : 0u);
    return e >= 94 ? m : (m >> min(94u - e, 31u));
}

// Exact mass of a bucket from its w sum, e its scores' exponent.
__device__ __forceinline__ u128 shifted_mass(unsigned long long wsum, int e) {
    const int s = e - 94;
    if (wsum == 0 || s <= 0) return wsum;
    if (s >= 64) return (u128)1 << 100;   // no score in [0, 1] has e > 127
    return (u128)wsum << s;
}

// Per-bucket sums of w: two 32-bit words (12-bit halves) or one 64-bit word.
template <bool kWide>
struct WSum {
    uint32_t *base;   // [2 * n] words
    int n;
    __device__ __forceinline__ void add(int d, uint32_t w) {
        if (kWide) {
            atomicAdd(reinterpret_cast<unsigned long long *>(base) + d, (unsigned long long)w);
        } else {
            atomicAdd(&base[d], w >> 12);
            atomicAdd(&base[n + d], w & 0xFFFu);
        }
    }
    __device__ __forceinline__ unsigned long long get(int d) const {
        if (kWide) return reinterpret_cast<const unsigned long long *>(base)[d];
        return ((unsigned long long)base[d] << 12) + base[n + d];
    }
};

// Visit scores 0..n-1 of one head with 16-byte loads when src is 16-byte
// aligned: thread tid reads vectors tid, tid + NT, ... (coalesced), four in
// flight.  f(k, v, in) is called for every lane, with in false past the end,
// so warp-wide votes inside f stay uniform.
template <int NT = kSelThreads, typename F>
__device__ __forceinline__ void for_scores4(const float *__restrict__ src, int n, bool vec, F f) {
    if (!vec) {
        for_scores<NT>(src, n, f);
        return;
    }
    const int tid = threadIdx.x;
    const int n4 = n >> 2;
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
    for (int base = 0; base < n4; base += 4 * NT) {
        float4 r[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = base + i * NT + tid;
            r[i] = k < n4 ? s4[k] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = base + i * NT + tid;
            const bool in = k < n4;
            f(4 * k, r[i].x, in);
            f(4 * k + 1, r[i].y, in);
            f(4 * k + 2, r[i].z, in);
            f(4 * k + 3, r[i].w, in);
        }
    }
    const int j = 4 * n4 + tid;   // at most three trailing scores
    f(j, j < n ? src[j] : 0.f, j < n);
}

// for_scores4 over global g that also copies every score into cache[0..n):
// the staging copy rides on the first histogram pass.
template <int NT = kSelThreads, typename F>
__device__ __forceinline__ void for_scores4_stage(const float *__restrict__ g, float *cache, int n,
                                                  F f) {
    const int tid = threadIdx.x;
    if ((reinterpret_cast<uintptr_t>(g) & 15) != 0) {
        for_scores<NT>(g, n, [&](int k, float v, bool in) {
            if (in) cache[k] = v;
            f(k, v, in);
        });
        return;
    }
    const int n4 = n >> 2;
    const float4 *g4 = reinterpret_cast<const float4 *>(g);
    float4 *c4 = reinterpret_cast<float4 *>(cache);
    for (int base = 0; base < n4; base += 4 * NT) {
        float4 r[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = base + i * NT + tid;
            r[i] = k < n4 ? g4[k] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = base + i * NT + tid;
            const bool in = k < n4;
            if (in) c4[k] = r[i];
            f(4 * k, r[i].x, in);
            f(4 * k + 1, r[i].y, in);
            f(4 * k + 2, r[i].z, in);
            f(4 * k + 3, r[i].w, in);
        }
    }
    const int j = 4 * n4 + tid;
    const float t = j < n ? g[j] : 0.f;
    if (j < n) cache[j] = t;
    f(j, t, j < n);
}

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(kPending) : "memory");
}

// for_scores4_stage with the copy done by cp.async: each thread copies its own
// 16-byte vectors (tid, tid + NT, ...) of a 16-byte aligned g into cache,
// eight in flight, one commit group per vector, and visits each as soon as
// its group has landed (a thread reads only what it copied itself, so no
// barrier is needed before the block's next one).
template <int NT = kSelThreads, typename F>
__device__ __forceinline__ void for_scores4_async(const float *__restrict__ g, float *cache, int n,
                                                  F f) {
    const int tid = threadIdx.x;
    const int n4 = n >> 2;
    const float4 *g4 = reinterpret_cast<const float4 *>(g);
    float4 *c4 = reinterpret_cast<float4 *>(cache);
    for (int base = 0; base < n4; base += 8 * NT) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int k = base + i * NT + tid;
            if (k < n4) cp_async16(c4 + k, g4 + k);
            cp_async_commit();
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i == 0) cp_async_wait<7>();
            if (i == 1) cp_async_wait<6>();
            if (i == 2) cp_async_wait<5>();
            if (i == 3) cp_async_wait<4>();
            if (i == 4) cp_async_wait<3>();
            if (i == 5) cp_async_wait<2>();
            if (i == 6) cp_async_wait<1>();
            if (i == 7) cp_async_wait<0>();
            const int k = base + i * NT + tid;
            const bool in = k < n4;
            const float4 r = in ? c4[k] : make_float4(0.f, 0.f, 0.f, 0.f);
            f(4 * k, r.x, in);
            f(4 * k + 1, r.y, in);
            f(4 * k + 2, r.z, in);
            f(4 * k + 3, r.w, in);
        }
    }
    const int j = 4 * n4 + tid;   // at most three trailing scores
    const float v = j < n ? g[j] : 0.f;
    if (j < n) cache[j] = v;
    f(j, v, j < n);
}

// Per-warp gather list: the warp appends the keys its lanes hit to its own
// segment of seg slots; n (the same in every lane) counts every hit, also
// those past seg that are not written.
struct WarpList {
    uint32_t *slot;
    int seg, n;
    __device__ __forceinline__ void append(bool hit, uint32_t key) {
        const unsigned msk = __ballot_sync(0xffffffffu, hit);
        if (hit) {
            const int p = n + __popc(msk & ((1u << (threadIdx.x & 31)) - 1u));
            if (p < seg) slot[p] = key;
        }
        n += __popc(msk);
    }
    __device__ __forceinline__ bool overflowed() const { return n > seg; }
};

// One head's MBA into mba[blockIdx.x] (written by thread 0 on every path).
template <bool kWide, int NT>
__device__ __forceinline__ void mba_head(uint8_t *sel_smem, const float *__restrict__ scores, int T,
                                         uint32_t num, uint32_t den, int cached, int list_cap,
                                         int32_t *__restrict__ mba, uint32_t *status) {
    uint32_t *hist = reinterpret_cast<uint32_t *>(sel_smem);   // [2 * 4096] w sums
    uint32_t *list = hist + 2 * kB0;                              // [list_cap] keys of d1
    float *cache = reinterpret_cast<float *>(list + list_cap);    // [T] when cached
    __shared__ u128 wt128[32], s_tot128;
    __shared__ unsigned long long wt64[32], s_tot64, s_add;
    __shared__ uint32_t s_cadd;
    __shared__ int s_d;
    const int tid = threadIdx.x, lane = tid & 31;
    const float *c = scores + (int64_t)blockIdx.x * T;
    const float *src = cached ? cache : c;
    const bool vec = cached || (reinterpret_cast<uintptr_t>(c) & 15) == 0;

    // 1. exact bucket masses (and the staging copy)
    WSum<kWide> W{hist, kB0};
    for (int i = tid; i < 2 * kB0; i += NT) hist[i] = 0u;
    if (tid == 0) s_d = -1;
    __syncthreads();
    int bad = 0;
    const auto body = [&](int, float v, bool in) {
        const bool valid = in && v >= 0.f && v <= 1.f;
        if (in && !valid) bad = 1;
        if (!valid) return;
        const uint32_t key = skey(v);
        W.add((int)(key >> 19), unit_mass(key));
    };
    if (cached && (reinterpret_cast<uintptr_t>(c) & 15) == 0)
        for_scores4_async<NT>(c, cache, T, body);
    else if (cached)
        for_scores4_stage<NT>(c, cache, T, body);
    else
        for_scores4<NT>(c, T, vec, body);
    __syncthreads();

    // 2. crossing bucket: thread t holds buckets 4095-4t .. 4092-4t (descending).
    // An invalid score adds 2^61, so one exact 128-bit total catches both it
    // and a head summing above 16.
    constexpr int kPer = kB0 / NT;   // buckets per thread
    u128 ml = bad ? (u128)1 << 61 : (u128)0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int d = kB0 - 1 - kPer * tid - i;
        ml += shifted_mass(W.get(d), d >> 4);
    }
    const u128 mpre = block_scan_excl(ml, wt128, &s_tot128);
    const u128 U128 = s_tot128;
    if (U128 > ((u128)1 << 60)) {   // invalid scores, or a head summing above 16
        if (tid == 0) {
            set_status(status, KVC_DEV_BAD_SCORE);
            mba[blockIdx.x] = 0;
        }
        return;
    }
    const unsigned long long U = (unsigned long long)U128;
    if (U == 0 || num == 0) {
        if (tid == 0) mba[blockIdx.x] = 0;
        return;
    }
    const u128 need = (u128)num * U;
    {
        // every partial sum is at most U <= 2^60 here
        unsigned long long run = (unsigned long long)mpre;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int d = kB0 - 1 - kPer * tid - i;
            const unsigned long long mi = (unsigned long long)shifted_mass(W.get(d), d >> 4);
            if (mi > 0 && (u128)den * run < need && (u128)den * (run + mi) >= need) {
                s_d = d;
                s_add = run;
            }
            run += mi;
        }
    }
    __syncthreads();
    const int d1 = s_d;
    if (d1 < 0) {   // unreachable: 0 < need <= den * U
        if (tid == 0) {
            set_status(status, KVC_DEV_BAD_SCORE);
            mba[blockIdx.x] = 0;
        }
        return;
    }
    unsigned long long A = s_add;
    const int e1 = d1 >> 4;   // exponent shared by every score of d1

    // 3. scores above d1 counted and d1's keys gathered; then the two
    // remaining digits (bits 18..9, 8..0) from the gathered keys
    uint32_t *cnt = hist;   // [1024] counts, then the w sums [2 * 1024]
    WSum<kWide> W2{hist + 1024, 1024};
    const int seg = list_cap / (NT / 32);
    WarpList wl{list + (tid >> 5) * seg, seg, 0};
    uint32_t cg = 0;
    for_scores4<NT>(src, T, vec, [&](int, float v, bool in) {
        const uint32_t key = skey(v);
        const int d = in ? (int)(key >> 19) : -1;
        cg += d > d1;
        wl.append(d == d1, key);
    });
    // the count above d1, with the number of overflowed warp lists in the high word
    const unsigned long long cgo = block_sum(
        (unsigned long long)cg | ((unsigned long long)(lane == 0 && wl.overflowed()) << 32), wt64,
        &s_tot64);
    uint32_t C = (uint32_t)cgo;
    const bool lists_ok = (cgo >> 32) == 0;
    uint32_t prefix = (uint32_t)d1;
    for (int pass = 1; pass < 3; ++pass) {
        const int bits = pass == 1 ? 10 : 9, shift = pass == 1 ? 9 : 0, nb = 1 << bits;
        // the digit's counts and masses from the gathered keys (all scores
        // if a list overflowed)
        for (int i = tid; i < 3 * 1024; i += NT) hist[i] = 0u;
        __syncthreads();
        const auto add = [&](uint32_t key) {
            if ((key >> (shift + bits)) != prefix) return;
            const int dd = (int)((key >> shift) & (uint32_t)(nb - 1));
            atomicAdd(&cnt[dd], 1u);
            W2.add(dd, unit_mass(key));
        };
        if (lists_ok) {
            for (int i = lane; i < wl.n; i += 32) add(wl.slot[i]);
        } else {
            for_scores4<NT>(src, T, vec, [&](int, float v, bool in) {
                if (in) add(skey(v));
            });
        }
        __syncthreads();
        // thread t holds buckets nb-1-per*t .. nb-per*(t+1) (descending),
        // each as its count in the high 64 bits and its mass (at most 2^60)
        // in the low 64 bits
        const int per = (nb + NT - 1) / NT;
        u128 pt = 0;
        for (int q = 0; q < per; ++q) {
            const int b = nb - 1 - per * tid - q;
            if (b >= 0) pt += shifted_mass(W2.get(b), e1) | ((u128)cnt[b] << 64);
        }
        u128 pp = block_scan_excl(pt, wt128, &s_tot128);
        for (int q = 0; q < per; ++q) {
            const int b = nb - 1 - per * tid - q;
            const u128 pb = b >= 0 ? shifted_mass(W2.get(b), e1) | ((u128)cnt[b] << 64) : (u128)0;
            const unsigned long long mb = (unsigned long long)pb, mp = (unsigned long long)pp;
            if (mb > 0 && (u128)den * (A + mp) < need && (u128)den * (A + mp + mb) >= need) {
                s_d = b;
                s_add = mp;
                s_cadd = (uint32_t)(pp >> 64);
            }
            pp += pb;
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
        const u128 have = (u128)den * A;
        const u128 step = (u128)den * ustar;
        long long m;
        if (step == 0 || have >= need) {
            set_status(status, KVC_DEV_BAD_SCORE);   // unreachable for valid scores
            m = C;
        } else {
            m = (long long)C + (long long)((need - have + step - 1) / step);
        }
        if (kDebugBounds && (m < 0 || m > T)) set_status(status, KVC_DEV_INVARIANT);
        mba[blockIdx.x] = (int32_t)m;
    }
}

// ------------------------------------------------------------------ budgets
// Computed by the last MBA block to finish, one thread per layer (L up to the
// block's threads, at most 1024).  Integer arithmetic only.
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

// Sum of v over the block (blockDim.x a multiple of 32, at most 1024); every
// thread receives it.  ws: 32 words of shared memory.
__device__ __forceinline__ unsigned long long block_add(unsigned long long v,
                                                        unsigned long long *ws) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) ws[warp] = v;
    __syncthreads();
    unsigned long long t = lane < (int)(blockDim.x >> 5) ? ws[lane] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    __syncthreads();
    return t;
}

// Largest-remainder split of R over the eligible layers by weight S (equal
// weights if the eligible weights sum to 0): every layer gets
// floor(R S_l / sum S); the leftover units go one each to the largest
// remainders, ties to the lower layer.  Returns the calling thread's share.
// red: 32 words of shared memory.
__device__ long long lr_split(int L, const long long *S, const unsigned char *elig, long long R,
                              long long *rem, unsigned long long *red) {
    const int l = threadIdx.x;
    const bool e = l < L && elig[l];
    unsigned long long sumw = block_add(e ? (unsigned long long)S[l] : 0ull, red);
    const unsigned long long n_el = block_add(e ? 1ull : 0ull, red);
    if (n_el == 0 || R <= 0) return 0;
    const bool equal = sumw == 0;
    if (equal) sumw = n_el;
    long long add = 0;
    unsigned long long q = 0, r = 0;
    if (e) {
        muldiv((unsigned long long)R, equal ? 1ull : (unsigned long long)S[l], sumw, q, r);
        add = (long long)q;
        rem[l] = (long long)r;
    }
    const long long left = R - (long long)block_add(q, red);
    if (e && left > 0) {
        long long rank = 0;
        for (int o = 0; o < L; ++o)
            rank += elig[o] && (rem[o] > rem[l] || (rem[o] == rem[l] && o < l));
        if (rank < left) add += 1;
    }
    __syncthreads();
    return add;
}

// Layer budgets from every head's MBA, by the block's first L threads (the
// block has at least L threads; every thread takes part in the barriers).
// S, rem: [kMaxLayers]; elig: [kMaxLayers]; red: [32] shared memory.
__device__ void layer_budgets(const int32_t *mba, int L, int Hkv, long long P, long long total,
                              long long floor_, int32_t *__restrict__ budget, uint32_t *status,
                              long long *S, long long *rem, unsigned char *elig,
                              unsigned long long *red) {
    const int l = threadIdx.x;
    const bool act = l < L;
    if (total >= (long long)L * P) {
        if (act) budget[l] = (int32_t)P;
        return;
    }
    if (act) {
        long long acc = 0;
        for (int k = 0; k < Hkv; ++k) acc += __ldcg(mba + (int64_t)l * Hkv + k);
        S[l] = acc;
        elig[l] = 1;
    }
    __syncthreads();
    long long B = floor_ + lr_split(L, S, elig, total - (long long)L * floor_, rem, red);
    while (true) {
        const long long over = act && B > P ? B - P : 0;
        if (over) B = P;
        const unsigned long long excess = block_add((unsigned long long)over, red);
        if (excess == 0) break;
        if (act) elig[l] = B < P;
        __syncthreads();
        B += lr_split(L, S, elig, (long long)excess, rem, red);
    }
    if (act) budget[l] = (int32_t)B;
    if (kDebugBounds) {   // sum = total (every layer at P if total >= L P), floor <= B <= P
        const unsigned long long sum = block_add(act ? (unsigned long long)B : 0ull, red);
        if (act && (B < floor_ || B > P)) set_status(status, KVC_DEV_INVARIANT);
        if (l == 0 && (long long)sum != total) set_status(status, KVC_DEV_INVARIANT);
    }
}

__device__ __forceinline__ unsigned long long warp_add(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// lr_split for L <= 32 by the whole block: lane l of every warp holds layer l
// and every warp computes the sums alike; warp w ranks layers w, w + (warps),
// ... with one ballot each, and the ranks meet in shared memory (rk: 32
// words).  The same arithmetic as lr_split.
__device__ long long lr_split_small(int L, long long S, bool e, long long R, long long *rk) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    e = e && lane < L;
    unsigned long long sumw = warp_add(e ? (unsigned long long)S : 0ull);
    const unsigned long long n_el = warp_add(e ? 1ull : 0ull);
    if (n_el == 0 || R <= 0) return 0;
    const bool equal = sumw == 0;
    if (equal) sumw = n_el;
    unsigned long long q = 0, r = 0;
    if (e) muldiv((unsigned long long)R, equal ? 1ull : (unsigned long long)S, sumw, q, r);
    const long long left = R - (long long)warp_add(q);
    // layers ranked before layer lw: larger remainder, or equal and lower index
    for (int lw = warp; lw < 32; lw += (int)(blockDim.x >> 5)) {
        const unsigned long long rw = __shfl_sync(0xffffffffu, r, lw);
        const unsigned before = __ballot_sync(0xffffffffu, e && (r > rw || (r == rw && lane < lw)));
        if (lane == 0) rk[lw] = __popc(before);
    }
    __syncthreads();
    const long long rank = rk[lane];
    __syncthreads();   // rk is rewritten by the next call
    long long add = (long long)q;
    if (e && left > 0 && rank < left) add += 1;
    return add;
}

// layer_budgets for L <= 32 by the whole block (lane l of every warp is layer
// l), the same arithmetic.  sh: 64 words of shared memory.
__device__ void layer_budgets_small(const int32_t *mba, int L, int Hkv, long long P,
                                    long long total, long long floor_,
                                    int32_t *__restrict__ budget, uint32_t *status, long long *sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool act = lane < L;
    if (total >= (long long)L * P) {
        if (threadIdx.x < L) budget[threadIdx.x] = (int32_t)P;
        return;
    }
    // S_l: warp l sums layer l's heads over its lanes
    for (int lw = warp; lw < L; lw += (int)(blockDim.x >> 5)) {
        unsigned long long acc = 0;
        for (int k = lane; k < Hkv; k += 32)
            acc += (unsigned long long)__ldcg(mba + (int64_t)lw * Hkv + k);
        acc = warp_add(acc);
        if (lane == 0) sh[32 + lw] = (long long)acc;
    }
    __syncthreads();
    const long long S = act ? sh[32 + lane] : 0;
    bool elig = act;
    long long B = floor_ + lr_split_small(L, S, elig, total - (long long)L * floor_, sh);
    while (true) {
        const long long over = act && B > P ? B - P : 0;
        if (over) B = P;
        const unsigned long long excess = warp_add((unsigned long long)over);
        if (excess == 0) break;
        elig = act && B < P;
        B += lr_split_small(L, S, elig, (long long)excess, sh);
    }
    if (threadIdx.x < L) budget[threadIdx.x] = (int32_t)B;
    if (kDebugBounds && warp == 0) {   // sum = total, floor <= B <= P
        const unsigned long long sum = warp_add(act ? (unsigned long long)B : 0ull);
        if (act && (B < floor_ || B > P)) set_status(status, KVC_DEV_INVARIANT);
        if (lane == 0 && (long long)sum != total) set_status(status, KVC_DEV_INVARIANT);
    }
}

// MBA of every head (one block each), then the layer budgets: the last block
// to finish (a completion counter in the workspace, reset by that block for
// the next launch; nothing waits on it) computes them from all heads' MBA.
template <bool kWide, int NT>
__global__ void __launch_bounds__(NT, 1024 / NT)
    mba_budget_kernel(const float *__restrict__ scores, int T, uint32_t num, uint32_t den,
                      int cached, int list_cap, int32_t *__restrict__ mba, int L, int Hkv,
                      long long P, long long total, long long floor_,
                      int32_t *__restrict__ budget, uint32_t *done, uint32_t *status) {
    extern __shared__ __align__(16) uint8_t sel_smem[];
    __shared__ int s_last;
    mba_head<kWide, NT>(sel_smem, scores, T, num, den, cached, list_cap, mba, status);
    __syncthreads();   // the head is done with shared memory; thread 0 wrote its MBA
    if (threadIdx.x == 0) {
        // release: this block's MBA is visible before the count moves;
        // acquire: the last block sees every other block's MBA
        uint32_t prev;
        asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(prev) : "l"(done) : "memory");
        s_last = prev == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (L <= 32) {
        layer_budgets_small(mba, L, Hkv, P, total, floor_, budget, status,
                            reinterpret_cast<long long *>(sel_smem));
        if (threadIdx.x == 0) *done = 0u;
        return;
    }
    long long *S = reinterpret_cast<long long *>(sel_smem);
    long long *rem = S + kMaxLayers;
    unsigned long long *red = reinterpret_cast<unsigned long long *>(rem + kMaxLayers);
    unsigned char *elig = reinterpret_cast<unsigned char *>(red + 32);
    layer_budgets(mba, L, Hkv, P, total, floor_, budget, status, S, rem, elig, red);
    if (threadIdx.x == 0) *done = 0u;
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
    __shared__ unsigned long long red[32];
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
        const long long over = act && B > P ? B - P : 0;
        if (over) B = P;
        const unsigned long long excess = block_add((unsigned long long)over, red);
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

// Writes the kept positions among one thread's 32 (bit i of gt: above v*,
// of eq: equal to v*; bit i stands for position j0 + i), G / E being the
// numbers above / equal to v* before the first of them: a kept position lands
// at G + min(E, need_eq), ties kept only while E < need_eq.
__device__ __forceinline__ void write_kept(uint32_t gt, uint32_t eq, int j0, int G, int E,
                                           int need_eq, long long B, int32_t *__restrict__ out) {
    for (uint32_t any = gt | eq; any; any &= any - 1u) {
        const int i = __ffs(any) - 1;
        if ((gt >> i) & 1u) {
            const int pos = G + (E < need_eq ? E : need_eq);
            if (pos >= 0 && pos < B) out[pos] = j0 + i;   // always true for valid scores
            ++G;
        } else {
            if (E < need_eq && G + E < B) out[G + E] = j0 + i;
            ++E;
        }
    }
}

__global__ void __launch_bounds__(kSelThreads)
    topk_kernel(const float *__restrict__ scores, int T, int P, int Hkv,
                const int32_t *__restrict__ budget, int per_head, int k_max, int cached,
                int staged, int list_cap, int32_t *__restrict__ idx, uint32_t *status) {
    extern __shared__ __align__(16) uint8_t sel_smem[];
    uint32_t *cnt = reinterpret_cast<uint32_t *>(sel_smem);   // [4096]
    uint32_t *list = cnt + kB0;                                 // [list_cap] keys of d1
    // the row ([P], when cached) or one compaction round of it ([32 * 1024],
    // when staged)
    float *cache = reinterpret_cast<float *>(list + list_cap);
    __shared__ uint32_t warp_tot[32];
    __shared__ uint32_t s_total, s_cadd;
    __shared__ unsigned long long wt64[32], s_tot64;
    __shared__ int s_d;
    const int head = blockIdx.x;
    const int l = head / Hkv;
    const int tid = threadIdx.x, lane = tid & 31;
    const float *c = scores + (int64_t)head * T;
    const float *src = cached ? cache : c;
    const bool vec = cached || (reinterpret_cast<uintptr_t>(c) & 15) == 0;
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
    // radix select of the B-th largest key: 12 bits (4096 buckets) over every
    // score (copying them into shared memory when they fit); the chosen
    // bucket's keys gathered into per-warp shared lists; then 10 and 9 bits
    // from the lists; each bucket search is a block-wide scan, one or four
    // buckets per thread
    for (int i = tid; i < kB0; i += kSelThreads) cnt[i] = 0;
    __syncthreads();
    int bad = 0;
    const auto body = [&](int, float v, bool in) {
        if (!in) return;
        if (!(v >= 0.f)) bad = 1;
        atomicAdd(&cnt[(skey(v) >> 19) & (kB0 - 1)], 1u);
    };
    if (cached && (reinterpret_cast<uintptr_t>(c) & 15) == 0)
        for_scores4_async(c, cache, P, body);
    else if (cached)
        for_scores4_stage(c, cache, P, body);
    else
        for_scores4(c, P, vec, body);
    bad = __syncthreads_or(bad);
    if (tid == 0 && bad) set_status(status, KVC_DEV_BAD_SCORE);
    // B is clamped to [1, P) above and P < 2^31: positions and counts from
    // here on are 32-bit
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
    const uint32_t d1 = (uint32_t)s_d;
    uint32_t prefix = d1;
    const int seg = list_cap / kSelWarps;
    WarpList wl{list + (tid >> 5) * seg, seg, 0};
    // Rows held in shared memory, and rows of at most four compaction rounds
    // (see below) copied round by round into a staging buffer: one pass marks
    // every position as above the chosen bucket (kept whatever v* is) or
    // inside it (decided once v* is known) in per-thread bit masks and gathers
    // the inside keys on the way.  Longer rows gather in a pass of their own.
    constexpr int kRound = 32 * kSelThreads;
    constexpr int kMaxRounds = 4;
    const bool merged = cached || (staged && P <= kMaxRounds * kRound);
    uint32_t above[kMaxRounds] = {0u, 0u, 0u, 0u}, inside[kMaxRounds] = {0u, 0u, 0u, 0u};
    if (merged) {
#pragma unroll
        for (int r = 0; r < kMaxRounds; ++r) {
            if (r * kRound >= P) break;
            const int n = min(P - r * kRound, kRound);   // positions of this round
            const float *rs = cache + r * kRound;
            if (!cached) {
                const float *g = c + r * kRound;
                if (vec) {
                    const float4 *g4 = reinterpret_cast<const float4 *>(g);
                    float4 *r4 = reinterpret_cast<float4 *>(cache);
                    for (int k = tid; k < (n >> 2); k += kSelThreads) r4[k] = g4[k];
                    for (int k = 4 * (n >> 2) + tid; k < n; k += kSelThreads) cache[k] = g[k];
                } else {
                    for (int k = tid; k < n; k += kSelThreads) cache[k] = g[k];
                }
                __syncthreads();
                rs = cache;
            }
            const int j0 = 32 * tid;   // within the round
            uint32_t ab = 0u, in = 0u;
            if (j0 + 32 <= n) {
                const float4 *s4 = reinterpret_cast<const float4 *>(rs + j0);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int q = (i + tid) & 7;   // rotated: distinct banks for 8 neighbours
                    const float4 v = s4[q];
                    const uint32_t e0 = skey(v.x) >> 19,
                                   e1 = skey(v.y) >> 19,
                                   e2 = skey(v.z) >> 19,
                                   e3 = skey(v.w) >> 19;
                    ab |= ((uint32_t)(e0 > d1) | ((uint32_t)(e1 > d1) << 1) |
                           ((uint32_t)(e2 > d1) << 2) | ((uint32_t)(e3 > d1) << 3)) << (4 * q);
                    in |= ((uint32_t)(e0 == d1) | ((uint32_t)(e1 == d1) << 1) |
                           ((uint32_t)(e2 == d1) << 2) | ((uint32_t)(e3 == d1) << 3)) << (4 * q);
                }
            } else {
                for (int i = 0; i < 32; ++i) {
                    if (j0 + i < n) {
                        const uint32_t e = skey(rs[j0 + i]) >> 19;
                        ab |= (uint32_t)(e > d1) << i;
                        in |= (uint32_t)(e == d1) << i;
                    }
                }
            }
            above[r] = ab;
            inside[r] = in;
            // the inside keys to this warp's list: slots from a warp prefix sum
            const int n_in = __popc(in);
            if (__any_sync(0xffffffffu, n_in != 0)) {
                int incl = n_in;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int a = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += a;
                }
                int slot = wl.n + incl - n_in;
                for (uint32_t m = in; m; m &= m - 1u, ++slot)
                    if (slot < seg) wl.slot[slot] = skey(rs[j0 + __ffs(m) - 1]);
                wl.n += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (!cached) __syncthreads();   // the next round's copy overwrites the buffer
        }
    } else {
        for_scores4(src, P, vec, [&](int, float v, bool in) {
            const uint32_t key = skey(v);
            wl.append(in && (key >> 19) == d1, key);
        });
    }
    const bool lists_ok = !__syncthreads_or(lane == 0 && wl.overflowed());
    for (int pass = 1; pass < 3; ++pass) {
        const int bits = pass == 1 ? 10 : 9, shift = pass == 1 ? 9 : 0, nb = 1 << bits;
        for (int i = tid; i < nb; i += kSelThreads) cnt[i] = 0;
        __syncthreads();
        const auto add = [&](uint32_t key) {
            if ((key >> (shift + bits)) == prefix)
                atomicAdd(&cnt[(key >> shift) & (uint32_t)(nb - 1)], 1u);
        };
        if (lists_ok) {
            for (int i = lane; i < wl.n; i += 32) add(wl.slot[i]);
        } else {   // a list overflowed: every score again
            for_scores4(src, P, vec, [&](int, float v, bool in) {
                if (in) add(skey(v));
            });
        }
        __syncthreads();
        const int b = nb - 1 - tid;   // thread t holds bucket nb-1-t (descending)
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
    // Ordered compaction in rounds of 32 scores per thread: thread t owns
    // positions base + 32t .. base + 32t + 31 and marks the ones above v* and
    // equal to v* in two bit masks; one block scan of the packed counts gives
    // each thread its first output slot.  Held rows reuse the masks of the
    // classification pass and reread only the inside positions; rows in
    // global memory are classified here (16-byte reads rotated by t so that
    // eight neighbouring threads hit distinct banks), each round first copied
    // into the (no longer needed) list area when it holds a whole round.
    const bool stage_rounds = !merged && !cached && list_cap >= kRound;
    int g_before = 0, e_before = 0;
    for (int base = 0; base < P; base += kRound) {
        const int j0 = base + 32 * tid;
        uint32_t gt = 0u, eq = 0u;
        if (merged) {
            const int r = base / kRound;
            gt = r == 0 ? above[0] : r == 1 ? above[1] : r == 2 ? above[2] : above[3];
            const uint32_t in =
                r == 0 ? inside[0] : r == 1 ? inside[1] : r == 2 ? inside[2] : inside[3];
            for (uint32_t m = in; m; m &= m - 1u) {
                const int i = __ffs(m) - 1;
                const uint32_t key = skey(cached ? cache[j0 + i] : c[j0 + i]);
                gt |= (uint32_t)(key > vstar) << i;
                eq |= (uint32_t)(key == vstar) << i;
            }
        } else {
            const int n = min(P - base, kRound);
            const float *rs = src + base;
            bool rvec = vec;
            if (stage_rounds) {
                float *rb = reinterpret_cast<float *>(list);
                if (vec) {
                    const float4 *g4 = reinterpret_cast<const float4 *>(rs);
                    float4 *r4 = reinterpret_cast<float4 *>(rb);
                    for (int k = tid; k < (n >> 2); k += kSelThreads) r4[k] = g4[k];
                    for (int k = 4 * (n >> 2) + tid; k < n; k += kSelThreads) rb[k] = rs[k];
                } else {
                    for (int k = tid; k < n; k += kSelThreads) rb[k] = rs[k];
                }
                __syncthreads();
                rs = rb;
                rvec = true;
            }
            const int r0 = 32 * tid;   // within the round
            if (rvec && r0 + 32 <= n) {
                const float4 *s4 = reinterpret_cast<const float4 *>(rs + r0);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int q = (i + tid) & 7;
                    const float4 r = s4[q];
                    const uint32_t k0 = skey(r.x), k1 = skey(r.y),
                                   k2 = skey(r.z), k3 = skey(r.w);
                    gt |= ((uint32_t)(k0 > vstar) | ((uint32_t)(k1 > vstar) << 1) |
                           ((uint32_t)(k2 > vstar) << 2) | ((uint32_t)(k3 > vstar) << 3))
                          << (4 * q);
                    eq |= ((uint32_t)(k0 == vstar) | ((uint32_t)(k1 == vstar) << 1) |
                           ((uint32_t)(k2 == vstar) << 2) | ((uint32_t)(k3 == vstar) << 3))
                          << (4 * q);
                }
            } else {
#pragma unroll 8
                for (int i = 0; i < 32; ++i) {
                    if (r0 + i < n) {
                        const uint32_t key = skey(rs[r0 + i]);
                        gt |= (uint32_t)(key > vstar) << i;
                        eq |= (uint32_t)(key == vstar) << i;
                    }
                }
            }
        }
        const unsigned long long packed = block_scan_excl(
            (unsigned long long)__popc(gt) | ((unsigned long long)__popc(eq) << 32), wt64,
            &s_tot64);
        write_kept(gt, eq, j0, g_before + (int)(uint32_t)packed, e_before + (int)(packed >> 32),
                   need_eq, B, out);
        const unsigned long long tot = s_tot64;
        g_before += (int)(uint32_t)tot;
        e_before += (int)(tot >> 32);
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

// Per device: the SM count and the dynamic shared memory a selection block
// may use alone on an SM (the block opt-in limit) or as one of two (half the
// SM's shared memory), each less 3 KiB for the kernels' static shared memory
// and the per-block reservation; the first call on a device raises the
// selection kernels' limit.
struct SelDevice {
    int sms = 0, smem_one = 0, smem_two_per_sm = 0;
};

SelDevice sel_device() {
    static std::mutex mu;
    static SelDevice cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SelDevice{};
    std::lock_guard<std::mutex> lk(mu);
    SelDevice &d = cache[dev];
    if (d.smem_one == 0) {
        int optin = 0, per_sm = 0, sms = 0;
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int lim = optin > 4096 ? optin - 2048 : 0;
        cudaFuncSetAttribute(mba_budget_kernel<false, 1024>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
        cudaFuncSetAttribute(mba_budget_kernel<true, 1024>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
        cudaFuncSetAttribute(mba_budget_kernel<false, 512>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
        // two of its blocks share an SM's shared memory
        cudaFuncSetAttribute(mba_budget_kernel<false, 512>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
        cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
        d.sms = sms;
        d.smem_two_per_sm = per_sm / 2 > 3072 ? min(per_sm / 2 - 3072, lim) : 0;
        d.smem_one = lim;
    }
    return d;
}

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

int launch_mba_budget(const kvc_shape &s, const float *scores, uint32_t num, uint32_t den,
                      int64_t total, int32_t floor_, int32_t *mba, int32_t *budget, uint32_t *done,
                      uint32_t *status, cudaStream_t st) {
    if (s.n_layers > kMaxLayers) {
        set_error("kvc_mba_budget: at most %d layers", kMaxLayers);
        return KVC_ERR_UNSUPPORTED;
    }
    const int heads = s.n_layers * s.n_kv_heads;
    const int T = s.seq_len;
    const SelDevice dev = sel_device();
    // Heads beyond one wave of 1024-thread blocks (one per SM): 512-thread
    // blocks, two per SM, with the rows read from L2 on each pass, when the
    // rows are short enough that 1024-thread blocks would hold them in shared
    // memory (longer rows: the 1024-thread form is faster) and the last block
    // has a thread per layer for the budgets.
    const bool half = heads > dev.sms && T <= kCacheFloats && s.n_layers <= 512;
    const int lim = half ? dev.smem_two_per_sm : dev.smem_one;
    const int hist = 2 * kB0 * 4;
    const int cached = T <= kCacheFloats && hist + T * 4 + kMinList * 4 <= lim;
    const int fixed = hist + (cached ? T * 4 : 0);
    if (fixed + kMinList * 4 > lim) {
        set_error("kvc_mba_budget: %d bytes of shared memory per block are too few", lim);
        return KVC_ERR_UNSUPPORTED;
    }
    const int list_cap = min(((lim - fixed) / 4) & ~3, (T + 3) & ~3);
    const size_t smem = (size_t)fixed + (size_t)list_cap * 4;
    const long long P = (long long)T - s.window;
    const bool wide = T > kSplitMaxT;
#define KVC_MBA_ARGS                                                                             \
    scores, T, num, den, cached, list_cap, mba, s.n_layers, s.n_kv_heads, P, (long long)total, \
        (long long)floor_, budget, done, status
    if (half)
        mba_budget_kernel<false, 512><<<heads, 512, smem, st>>>(KVC_MBA_ARGS);
    else if (!wide)
        mba_budget_kernel<false, 1024><<<heads, 1024, smem, st>>>(KVC_MBA_ARGS);
    else
        mba_budget_kernel<true, 1024><<<heads, 1024, smem, st>>>(KVC_MBA_ARGS);
#undef KVC_MBA_ARGS
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_mba_budget: launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

int launch_topk(const kvc_shape &s, const float *scores, const int32_t *budget, int per_head,
                int32_t k_max, int32_t *idx, uint32_t *status, cudaStream_t st) {
    const int heads = s.n_layers * s.n_kv_heads;
    const int P = s.seq_len - s.window;
    const int lim = sel_device().smem_one;
    const int hist = kB0 * 4;
    const int cached = P <= kCacheFloats && hist + P * 4 + kMinList * 4 <= lim;
    // rows of at most four compaction rounds that are not held whole: a
    // one-round staging buffer
    const int round = 32 * kSelThreads;
    const int staged = !cached && P <= 4 * round && hist + round * 4 + kMinList * 4 <= lim;
    const int fixed = hist + (cached ? P * 4 : staged ? round * 4 : 0);
    if (fixed + kMinList * 4 > lim) {
        set_error("kvc_topk_select: %d bytes of shared memory per block are too few", lim);
        return KVC_ERR_UNSUPPORTED;
    }
    const int list_cap = min(((lim - fixed) / 4) & ~3, (P + 3) & ~3);
    const size_t smem = (size_t)fixed + (size_t)list_cap * 4;
    topk_kernel<<<heads, kSelThreads, smem, st>>>(scores, s.seq_len, P, s.n_kv_heads, budget,
                                                   per_head, k_max, cached, staged, list_cap, idx,
                                                   status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kvc_topk_select: launch failed: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

}  // namespace kvc
