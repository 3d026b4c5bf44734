// kvc_internal.cuh -- definitions shared by the libkvc translation units:
// workspace layout, the score-pass work split, and thin inline-PTX wrappers
// for the sm_100-family async machinery (mbarrier, TMA, tcgen05/TMEM).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "../../include/kvc.h"

namespace kvc {

// ---------------------------------------------------------------- constants
constexpr int kTileKeys = 128;          // keys per score tile of the CUDA-core path
constexpr int kPairKeys = 256;          // keys per SM-pair tile of the tensor-core path
constexpr int kMaxRowsTC = 512;         // G*W handled by the tensor-core path
constexpr size_t kWsHeader = 256;       // status word, MBA completion counter, padding
constexpr double kLog2e = 1.4426950408889634;

// Every pipeline wait gives up after this many nanoseconds of %globaltimer,
// sets KVC_DEV_TIMEOUT and lets the kernel unwind.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;
// A waiting thread is suspended in hardware until the barrier's phase
// completes or this many nanoseconds pass (then the limit above is checked):
// far fewer polling instructions than a spin.
#define KVC_SUSPEND_HINT_NS "10000000"

// ---------------------------------------------------------------- score split
// The score passes walk the flat sequence of (unit, key-tile) pairs, unit =
// (layer, KV head), in unit-major order.  Worker c of g (a CTA on the CUDA
// cores, a 2-CTA cluster on the tensor cores) owns tiles [floor(N c / g),
// floor(N (c+1) / g)).  Pass 1 leaves one partial (max, sum) per row for
// every (unit, worker touching it) in slot c - first_worker(unit).
struct ScoreSplit {
    int64_t n_units;       // L * H_kv
    int64_t tiles_per_unit;
    int64_t n_tiles;       // n_units * tiles_per_unit
    int grid;              // workers: CTAs, or CTA pairs on the tensor-core path
    int max_slots;         // partial slots per unit
    int rows;              // G * W
    int rows_pad;          // rows rounded up to 128 (CUDA cores) or 256 (tensor cores)
};

__host__ __device__ inline int64_t split_begin(int64_t n, int g, int64_t c) {
    return (n * c) / g;
}
__host__ __device__ inline int64_t split_cta_of(int64_t n, int g, int64_t t) {
    return ((int64_t)g * (t + 1) - 1) / n;
}

// tc: 256-key tiles over `pairs` CTA pairs; otherwise 128-key tiles over
// four CTAs per SM.
inline ScoreSplit make_score_split(const kvc_shape &s, bool tc, int sms, int pairs) {
    ScoreSplit sp;
    const int G = s.n_q_heads / s.n_kv_heads;
    const int tile = tc ? kPairKeys : kTileKeys;
    sp.n_units = (int64_t)s.n_layers * s.n_kv_heads;
    sp.tiles_per_unit = (s.seq_len + tile - 1) / tile;
    sp.n_tiles = sp.n_units * sp.tiles_per_unit;
    const int64_t want = tc ? (pairs > 0 ? pairs : 1) : 4LL * (sms > 0 ? sms : 148);
    sp.grid = (int)(sp.n_tiles < want ? sp.n_tiles : want);
    sp.rows = G * s.window;
    const int rb = tc ? 256 : 128;
    sp.rows_pad = (sp.rows + rb - 1) / rb * rb;
    int mx = 1;
    for (int64_t u = 0; u < sp.n_units; ++u) {
        const int64_t a = split_cta_of(sp.n_tiles, sp.grid, u * sp.tiles_per_unit);
        const int64_t b = split_cta_of(sp.n_tiles, sp.grid, u * sp.tiles_per_unit + sp.tiles_per_unit - 1);
        if (b - a + 1 > mx) mx = (int)(b - a + 1);
    }
    sp.max_slots = mx;
    return sp;
}

// Bounds-checking build (nvcc -DKVC_DEBUG_BOUNDS): kernels verify their
// outputs' invariants and OR KVC_DEV_INVARIANT into the status word on a
// failure, without trapping; the checks compile away otherwise.
#ifdef KVC_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif

// ---------------------------------------------------------------- status word
__device__ __forceinline__ void set_status(uint32_t *status, uint32_t bits) {
    atomicOr(status, bits);
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, " KVC_SUSPEND_HINT_NS ";\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity.  Returns false (and
// records KVC_DEV_TIMEOUT / raises the CTA abort flag) if the limit passes,
// or immediately if another thread of the CTA already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          uint32_t *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            set_status(status, KVC_DEV_TIMEOUT);
            return false;
        }
    }
}

// The same bounded wait with acquire at cluster scope, for barriers that
// other CTAs of the cluster arrive on.
__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, " KVC_SUSPEND_HINT_NS ";\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cl(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                             uint32_t *status) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait_cl(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            set_status(status, KVC_DEV_TIMEOUT);
            return false;
        }
    }
}

// Wait used only while unwinding: bounded, ignores the abort flag.
__device__ __forceinline__ bool mbar_drain(uint64_t *bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() - t0 > kWaitLimitNs) return false;
    return true;
}

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address, in the cluster's shared window, of the object at shared-memory
// address `saddr` of CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// Arrive on an mbarrier given by its cluster address.  The plain form
// releases at CTA scope, enough when the arriving thread's own work is
// already complete (a finished TMEM load, an observed TMA completion) and
// cheap; the _cluster form orders the thread's earlier shared-memory writes
// for readers in the other CTA and costs a cluster-scope fence.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load; c0 is the innermost coordinate (must be a multiple of
// 16 bytes' worth of elements).
__device__ __forceinline__ void tma_load_3d(const CUtensorMap *map, uint64_t *bar, void *dst, int c0,
                                            int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand stored in the
// 128-byte swizzled layout that TMA writes for a box whose inner extent is
// 128 bytes: 8-row groups of 1024 bytes (stride-dimension offset 1024).
// Bits: [0,14) start>>4, [16,30) leading offset>>4 (unused for this layout),
// [32,46) stride offset>>4, [46,48) descriptor version 1, [61,64) layout 2 =
// 128-byte swizzle.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B, fp32 accumulator,
// both operands K-major: [4,6) D format (1 = f32), [7,10) A format (1 =
// bf16), [10,13) B format (1 = bf16), [17,23) N>>3, [24,29) M>>4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// SM-pair forms (cta_group::2): TMEM is allocated in both CTAs of a 2-CTA
// cluster by one warp of each; one thread of the even CTA issues M = 256
// MMAs whose A rows 0-127 and B rows 0..N/2-1 come from the even CTA's
// shared memory and the rest from the odd CTA's at the same offsets, each
// CTA's TMEM receiving its own 128 rows of D; a commit arrives on the
// barrier at the same offset in every CTA of the mask.  A kernel uses
// either these forms or the single-CTA ones, never both.
__device__ __forceinline__ void tmem_alloc2(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_mma2_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit2(uint64_t *bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// The SM-pair MMA with its A operand in TMEM (one 128-lane block per CTA at
// the same TMEM address in both) and B from shared memory.
__device__ __forceinline__ void tc_mma2_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                    uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 registers -> 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
// 16 registers -> 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 lanes x 32 consecutive columns of 32-bit TMEM cells -> 32 registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Compiler-level fence: uses of v cannot be scheduled before this point
// (place it right after tmem_ld_wait, which orders it after the hardware
// wait).  tcgen05.ld writes its registers asynchronously.
__device__ __forceinline__ void reg_fence(float (&v)[32]) {
    asm volatile(""
                 : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                   "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]),
                   "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15]), "+f"(v[16]), "+f"(v[17]),
                   "+f"(v[18]), "+f"(v[19]), "+f"(v[20]), "+f"(v[21]), "+f"(v[22]), "+f"(v[23]),
                   "+f"(v[24]), "+f"(v[25]), "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]),
                   "+f"(v[30]), "+f"(v[31]));
}

// Hardware base-2 exponential (PTX ex2.approx.ftz.f32; ex2(-inf) = +0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed pairs of fp32 (sm_100-family f32x2 ALU forms): one instruction
// operates on two floats held in a 64-bit register pair.
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long r, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// max of three floats in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- Keyformer noise
// (both score paths draw the same numbers for the same (unit, row, key)):
// key j of row r takes word j mod 4 of the Philox4x32-10 block (Salmon et
// al., "Parallel random numbers: as easy as 1, 2, 3", SC 2011) at counter
// (j / 4, r, unit, 0), so one block serves four consecutive keys of a row.
__device__ __forceinline__ void philox4(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t k0,
                                        uint32_t k1, uint32_t (&o)[4]) {
    uint32_t c3 = 0;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    o[0] = c0;
    o[1] = c1;
    o[2] = c2;
    o[3] = c3;
}

// Word s (0..3, a run-time value) of a block.
__device__ __forceinline__ uint32_t pick4(const uint32_t (&o)[4], uint32_t s) {
    const uint32_t a = (s & 1) ? o[1] : o[0], b = (s & 1) ? o[3] : o[2];
    return (s & 2) ? b : a;
}

// Gumbel draw from a 32-bit word: u = (b + 1/2) 2^-24 from its top 24 bits
// b, zeta = -ln(-ln u).  -ln u is formed from whichever of u and 1 - u is
// exact in fp32 (log1p near 1), so the rare draws close to 1 -- the large
// zeta that dominate a row -- come out accurately.
__device__ __forceinline__ float gumbel_bits(uint32_t w) {
    const uint32_t b = w >> 8;
    float nlu;
    if (b >= (1u << 23)) {
        const float v = ((float)((1u << 24) - 1u - b) + 0.5f) * 0x1p-24f;   // 1 - u, exact
        nlu = -log1pf(-v);
    } else {
        const float u = ((float)b + 0.5f) * 0x1p-24f;                       // exact
        nlu = -logf(u);
    }
    return -logf(nlu);
}

// One draw for (unit, row, key) (a whole block for one word: the CUDA-core
// path; the tensor-core epilogues use every word of each block).
__device__ __forceinline__ float gumbel(uint32_t unit, uint32_t row, uint32_t key, uint32_t k0,
                                        uint32_t k1) {
    uint32_t o[4];
    philox4(key >> 2, row, unit, k0, k1, o);
    return gumbel_bits(pick4(o, key & 3));
}

// ---------------------------------------------------------------- host side
struct ScoreArgs {
    const void *q;
    const void *k;
    float *scores;
    float2 *partial;   // [units][max_slots][rows_pad] (running max, sum), log2 units
    float *neg_bias;   // [units][rows_pad] = -(max + log2(sum)), -inf for pad rows
    uint32_t *status;
    bool stats_only = false;   // stop after pass 1 + merge (row biases only)
};

// CTA pairs of the tensor-core score kernels that the current device runs at
// once (cached per device; half the SM count if the query fails).
int score_tc_pairs(int sms);
// 3-D bf16 TMA view [outer][mid][inner] with a (64, box_rows, 1) box and the
// 128-byte swizzle; rows past `mid` read as zeros.  False if the driver
// entry point is missing or the encoding is refused.
bool make_tma_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t mid, uint64_t outer,
                  uint32_t box_rows);
int launch_score_tc(const kvc_shape &s, const ScoreSplit &sp, const ScoreArgs &a, cudaStream_t st);
int launch_score_tc_keyformer(const kvc_shape &s, const ScoreSplit &sp, const ScoreArgs &a,
                              uint64_t seed, double tau, cudaStream_t st);
int launch_score_simt(const kvc_shape &s, const ScoreSplit &sp, const ScoreArgs &a,
                      cudaStream_t st);
int launch_score_merge(const kvc_shape &s, const ScoreSplit &sp, const ScoreArgs &a,
                       cudaStream_t st);
int launch_score_keyformer(const kvc_shape &s, const ScoreSplit &sp, const ScoreArgs &a,
                           uint64_t seed, double tau, cudaStream_t st);
// MBA of every head and the layer budgets in one launch; done is a workspace
// word that is zero between launches.
int launch_mba_budget(const kvc_shape &s, const float *scores, uint32_t num, uint32_t den,
                      int64_t total, int32_t floor_, int32_t *mba, int32_t *budget, uint32_t *done,
                      uint32_t *status, cudaStream_t st);
// per_head == 0: budget[L] per layer; 1: budget[L][H_kv] per head.
int launch_topk(const kvc_shape &s, const float *scores, const int32_t *budget, int per_head,
                int32_t k_max, int32_t *idx, uint32_t *status, cudaStream_t st);
int launch_head_budget(const kvc_shape &s, const int32_t *mba, const int32_t *budget,
                       int32_t *head_budget, cudaStream_t st);
int launch_threshold(const kvc_shape &s, const float *scores, float tau, int32_t k_max,
                     int32_t *idx, int32_t *counts, uint32_t *status, cudaStream_t st);
int launch_pool(const kvc_shape &s, const float *scores, int32_t kernel, int32_t mode, float *pooled,
                cudaStream_t st);
int launch_compact(const kvc_shape &s, const void *k, const void *v, const int32_t *idx,
                   const int32_t *budget, int per_head, int32_t k_max, void *k_out, void *v_out,
                   int64_t out_rows, uint32_t *status, cudaStream_t st);
// q == nullptr: magnitude criterion; otherwise the query-driven one.  With
// `given` ([L][H_kv][D] fp32) the channels are ranked by those scores instead
// (THINKV), and k_out may be any packed cache (the compacted values).
int launch_channel_prune(const kvc_shape &s, const void *q, const void *k_out, const int32_t *budget,
                         int32_t keep, int32_t *chan, void *k_pruned, int64_t pruned_elems,
                         uint32_t *status, cudaStream_t st, const float *given = nullptr);
// THINKV: per-channel value scores [L][H_kv][D] (fp32 sums of squared window
// attention outputs) from the row biases that a stats-only score pass left
// in a.neg_bias; `partial` is scratch of value_partial_floats() floats.
constexpr int kValueTcParts = 16;  // (job, CTA, warp) partial sums per unit, tensor-core kernel
int64_t value_partial_floats(const kvc_shape &s);
// The tensor-core THINKV kernel serves bf16, head_dim 128, G*W <= 512.
bool value_tc_eligible(const kvc_shape &s);
int launch_value_tc(const kvc_shape &s, const ScoreSplit &sp, const void *q, const void *k,
                    const void *v, const float *neg_bias, float *partial, uint32_t *status,
                    cudaStream_t st, int *parts_out);
int launch_value_scores(const kvc_shape &s, const ScoreSplit &sp, const void *q, const void *k,
                        const void *v, const float *neg_bias, float *partial, float *score_v,
                        bool tc, uint32_t *status, cudaStream_t st);

void set_error(const char *fmt, ...);

// One NVTX range per C-ABI call, named after the call, around its host-side
// work (validation and enqueueing): a profiler's timeline shows which call
// launched which kernels.  Without a profiler attached the push and pop are a
// check of an unset function pointer.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

// Shared by every scoring entry point (api.cu): shape validation (message in
// kvc_last_error on failure), whether the tensor-core kernels can serve the
// shape on the current device, the KVC_SCORE_IMPL choice (0 auto, 1 simt,
// 2 tc, -1 invalid) and the work split for the current device.
bool shape_ok(const kvc_shape *s, const char *fn);
bool tc_eligible(const kvc_shape &s);
int score_impl_choice();
ScoreSplit make_split(const kvc_shape &s, bool tc);

}  // namespace kvc
