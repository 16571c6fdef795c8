// Device helpers for the sm_103a kernels: mbarriers, TMA, tcgen05 (UMMA +
// TMEM), shared-memory matrix descriptors and bounded waits.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

constexpr int kD = 512;          // latent width
constexpr int kP = 64;           // shared rotary key width
constexpr int kW = 576;          // values per cached token
constexpr int kRowBf16 = 1152;   // bytes per bf16 row
constexpr int kRowFp8 = 656;     // bytes per fp8_ds_mla row
constexpr int kTile = 128;       // tokens per decode tile (UMMA M)

// Device-side status bits written to the first word of the decode workspace.
constexpr int kErrWaitTimeout = 1;   // a bounded wait gave up
constexpr int kErrBadBlock = 2;      // a block-table entry pointed outside the pool
constexpr int kErrF16Range = 4;      // fp8 rows: a block scale or query value beyond the f16 range

// A wait that never ends would hold the GPU; every spin gives up after this.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Busy-waits about `ns` nanoseconds of %globaltimer (test hooks only).
static __device__ __noinline__ void spin_for_ns(unsigned long long ns) {
    const unsigned long long t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < ns) {
    }
}

// ------------------------------------------------------------- mbarriers

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, "
        "p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Slow path of the waits below: spins until the phase completes, `abort` is
// raised by another role, or kWaitLimitNs passes (returns false then).
template <bool kCluster>
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort) {
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        uint32_t ok;
        if (kCluster)
            asm volatile(
                "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}"
                : "=r"(ok)
                : "r"(smem_u32(bar)), "r"(parity)
                : "memory");
        else
            asm volatile(
                "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}"
                : "=r"(ok)
                : "r"(smem_u32(bar)), "r"(parity)
                : "memory");
        if (ok) return true;
        if ((i & 63) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
        }
    }
}

// Waits for the phase of `bar` with the given parity to complete (bounded).
// The first probe is inline and needs no call, so an already-completed phase
// costs a single instruction.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow<false>(bar, parity, abort);
}

// Same, with cluster-scope acquire: for barriers completed by another CTA of
// the cluster (remote arrivals or st.async transactions into this CTA).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    return mbar_wait_slow<true>(bar, parity, abort);
}

// ------------------------------------------------------------------ cluster

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared-memory address (shared::cluster window) of the same offset in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Reads the int at the offset of `flag` in CTA `rank` of the cluster.
__device__ __forceinline__ int peer_aborted(volatile int* flag, uint32_t rank) {
    int v;
    asm volatile("ld.shared::cluster.relaxed.cluster.s32 %0, [%1];" : "=r"(v)
                 : "r"(mapa_shared(smem_u32(const_cast<int*>(flag)), rank))
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Asynchronous 16-byte store into another CTA's shared memory that counts its
// bytes as a transaction on that CTA's mbarrier (both cluster addresses).
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
        "r"(a), "r"(b), "r"(c), "r"(d), "r"(remote_bar)
        : "memory");
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from this CTA's shared memory into another CTA's (cluster address), counted
// as a transaction on that CTA's mbarrier.
__device__ __forceinline__ void bulk_s2cluster(uint32_t dst_cluster, const void* src, uint32_t bytes,
                                               uint32_t remote_bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst_cluster),
        "r"(smem_u32(src)), "r"(bytes), "r"(remote_bar)
        : "memory");
}

// Arrive on an mbarrier in another CTA of the cluster without ordering this
// thread's earlier memory operations (a release at cluster scope would wait
// for its in-flight remote stores, about a microsecond). Used only to hand a
// buffer back after reads whose values have already been consumed.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Programmatic dependent launch: a grid launched with programmatic stream
// serialisation may start before the previous kernel in the stream ends;
// griddep_wait() blocks until that kernel has finished and its writes are
// visible. griddep_launch_dependents() lets the next such grid start early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ proxies

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Block-subset barrier that also returns the OR of `pred` over the threads.
__device__ __forceinline__ int named_bar_or(int id, int nthreads, int pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.s32 %0, 1, 0, "
        "q;\n\t}"
        : "=r"(r)
        : "r"(pred), "r"(id), "r"(nthreads)
        : "memory");
    return r;
}

// Block-subset barrier that returns the AND of `pred` over the threads.
__device__ __forceinline__ int named_bar_and(int id, int nthreads, int pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\tselp.s32 %0, 1, 0, "
        "q;\n\t}"
        : "=r"(r)
        : "r"(pred), "r"(id), "r"(nthreads)
        : "memory");
    return r;
}

// ---------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// tma_load_2d delivered to every CTA of the cluster named in cta_mask, at the
// same shared-memory offset, each copy counted on that CTA's mbarrier at the
// offset of `bar`.
__device__ __forceinline__ void tma_load_2d_mc(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                               uint16_t cta_mask, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5, %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "h"(cta_mask), "l"(policy)
        : "memory");
}

// Bulk prefetch of [addr, addr + bytes) into L2 (bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void* addr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(addr)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D(tmem) (+)= A(smem desc) * B(smem desc), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D(tmem) (+)= A(tmem) * B(smem desc), bf16 inputs, fp32 accumulate. A is
// M x 16 at column a_tmem: row m in lane m, two bf16 values a column (the
// lower k in the low half), K-major.
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// umma_commit that arrives on the mbarrier at the offset of `bar` in every
// CTA of the cluster named in cta_mask.
__device__ __forceinline__ void umma_commit_mc(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Waits (bounded, whatever the abort flag says) until every tcgen05.mma this
// thread has issued is complete, through a one-use mbarrier of count 1.
__device__ __forceinline__ void drain_mma(uint64_t* bar) {
    umma_commit(bar);
    volatile int never = 0;
    mbar_wait(bar, 0, &never);
}

#include "tmem_ldst.inc"

// Shared-memory matrix descriptor (sm_100 family layout):
//   [0,14) start >> 4, [16,30) leading byte offset >> 4, [32,46) stride byte
//   offset >> 4, [46,48) = 1, [61,64) swizzle mode.
enum SwizzleMode : uint32_t { kSwNone = 0, kSw128 = 2, kSw64 = 4, kSw32 = 6 };

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t mode) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(mode & 7u) << 61;
    return d;
}

// Instruction descriptor for kind::f16 with bf16 (or f16) A/B and fp32 D.
//   [4,6) D format (1 = f32), [7,10) A format (0 = f16, 1 = bf16), [10,13) B
//   format, bit 15 A major (1 = MN), bit 16 B major, [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major, bool f16 = false) {
    return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// 4 x 4 transpose inside each quad of lanes: lane 4j + k holds in x[c]
// column c of row k; afterwards it holds column k of rows 0..3 (x[r] = row r).
// Two butterfly stages of two shuffles each, then a reorder by the lane bits.
__device__ __forceinline__ void quad_transpose(float (&x)[4], int lane) {
    const bool b1 = (lane & 2) != 0, b0 = (lane & 1) != 0;
    // rows k and k ^ 2 trade the column pair the other keeps
    const float s0 = b1 ? x[0] : x[2], s1 = b1 ? x[1] : x[3];
    const float k0 = b1 ? x[2] : x[0], k1 = b1 ? x[3] : x[1];
    const float r0 = __shfl_xor_sync(0xffffffffu, s0, 2), r1 = __shfl_xor_sync(0xffffffffu, s1, 2);
    // rows k and k ^ 1 trade the column the other keeps
    const float t0 = b0 ? k0 : k1, t1 = b0 ? r0 : r1;
    const float m0 = b0 ? k1 : k0, m1 = b0 ? r1 : r0;
    const float u0 = __shfl_xor_sync(0xffffffffu, t0, 1), u1 = __shfl_xor_sync(0xffffffffu, t1, 1);
    // column k of rows k, k ^ 1, k ^ 2, k ^ 3 is m0, u0, m1, u1: put row r at x[r]
    const float w0 = b0 ? u0 : m0, w1 = b0 ? m0 : u0, w2 = b0 ? u1 : m1, w3 = b0 ? m1 : u1;
    x[0] = b1 ? w2 : w0;
    x[1] = b1 ? w3 : w1;
    x[2] = b1 ? w0 : w2;
    x[3] = b1 ? w1 : w3;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// e4m3 x16 (one uint4) times a scale -> 16 f16 (two uint4): each code widens
// exactly to f16, one f16 multiply (round to nearest even) by the scale
// rounded to f16. |code| <= 448, so a scale up to 146 keeps every product
// finite.
__device__ __forceinline__ void dequant16_h(uint4 codes, __half2 sc, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] & 0xFFFFu), __NV_E4M3);
        const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] >> 16), __NV_E4M3);
        const __half2 p01 = __hmul2(*reinterpret_cast<const __half2*>(&h01), sc);
        const __half2 p23 = __hmul2(*reinterpret_cast<const __half2*>(&h23), sc);
        o[2 * i] = *reinterpret_cast<const uint32_t*>(&p01);
        o[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&p23);
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// e4m3 x16 (one uint4) times scale -> 16 bf16 (two uint4): each code widens
// exactly (e4m3 -> half -> float), one fp32 multiply, round to nearest even.
__device__ __forceinline__ void dequant16(uint4 codes, float scale, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] & 0xFFFFu), __NV_E4M3);
        const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] >> 16), __NV_E4M3);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
        o[2 * i] = pack_bf16x2(f01.x * scale, f01.y * scale);
        o[2 * i + 1] = pack_bf16x2(f23.x * scale, f23.y * scale);
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

}  // namespace mla
