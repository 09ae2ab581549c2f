// Device helpers shared by the kernels of libcolibri.so (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "colibri.h"

namespace clb {

constexpr int G = COLIBRI_GROUP;  // quantisation group
constexpr unsigned FULL = 0xffffffffu;

// Error bits written to the workspace flag.
constexpr int ERR_BAD_ID = 1;       // an expert id outside [0, E)
constexpr int ERR_WAIT_TIMEOUT = 2; // an mbarrier or flag wait ran out of iterations
constexpr int ERR_BAD_SHAPE = 4;    // a kernel was handed a shape it does not cover

// Bound on any wait in these kernels: a wait gives up (and its kernel reports
// ERR_WAIT_TIMEOUT) after WAIT_LIMIT_NS of global time, far beyond any legal wait.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
// Suspend-time hint of one mbarrier try_wait: the thread sleeps until the phase completes
// or this much time passes, instead of spinning on the issue slots.
constexpr uint32_t WAIT_HINT_NS = 1000000u;

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// One-use loads of weight bytes: bypass L1, they are read once per call.
__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_nc(const void *p)
{
    return __ldg(reinterpret_cast<const uint4 *>(p));
}


// sum of four unsigned bytes of a times four signed bytes of b, plus c
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// The 16 bytes of one 32-element group of offset-binary nibbles (byte j: element 2j in
// the low nibble, 2j+1 in the high nibble), split without shifting: l[i] keeps the low
// nibbles (elements 8i, 8i+2, 8i+4, 8i+6) as bytes, h[i] the high nibbles as 16x their
// value (elements 8i+1, ..., 8i+7).
struct NibbleSplit {
    uint32_t l[4], h[4];
};

__device__ __forceinline__ NibbleSplit split_nibbles(uint4 w)
{
    constexpr uint32_t LO = 0x0F0F0F0Fu, HI = 0xF0F0F0F0u;
    NibbleSplit n;
    n.l[0] = w.x & LO, n.h[0] = w.x & HI;
    n.l[1] = w.y & LO, n.h[1] = w.y & HI;
    n.l[2] = w.z & LO, n.h[2] = w.z & HI;
    n.l[3] = w.w & LO, n.h[3] = w.w & HI;
    return n;
}

// int32 dot of one group against activation codes stored as 8 words in even/odd order
// (word 2i = elements 8i, 8i+2, 8i+4, 8i+6; word 2i+1 = elements 8i+1, ..., 8i+7), given
// corr = 8 * (sum of the 32 codes), which removes the +8 offset of the nibbles. The sum
// over the high nibbles carries a factor 16 and is a multiple of 16, so the arithmetic
// shift by 4 is exact.
__device__ __forceinline__ int dot_split(const NibbleSplit &n, uint4 a0, uint4 a1, int corr)
{
    int lo = dp4a_us(n.l[0], a0.x, 0);
    int hi = dp4a_us(n.h[0], a0.y, 0);
    lo = dp4a_us(n.l[1], a0.z, lo);
    hi = dp4a_us(n.h[1], a0.w, hi);
    lo = dp4a_us(n.l[2], a1.x, lo);
    hi = dp4a_us(n.h[2], a1.y, hi);
    lo = dp4a_us(n.l[3], a1.z, lo);
    hi = dp4a_us(n.h[3], a1.w, hi);
    return lo + (hi >> 4) - corr;
}

// Byte position of element k (0..31) of a group in the even/odd word order.
__device__ __forceinline__ int eo_pos(int k)
{
    return (k & ~7) + ((k & 1) ? 4 + ((k & 7) >> 1) : ((k & 7) >> 1));
}

// Position of element k (0..31) of a group in the tensor-core k order: inside each run of
// 8 elements, slot s holds element (0, 4, 1, 5, 2, 6, 3, 7)[s], the order in which the
// prefill converters unpack a 32-bit word of eight nibbles into four bf16 pairs.
__host__ __device__ __forceinline__ int bf16_pos(int k)
{
    return (k & ~7) + ((k & 3) << 1) + ((k >> 2) & 1);
}

// bf16 bit pattern of a small integer (exact for |q| <= 256): the upper half of the fp32
// pattern of (float)q.
__device__ __forceinline__ uint16_t bf16_of_int(int q)
{
    return (uint16_t)(__float_as_uint((float)q) >> 16);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(FULL, v, o);
    return v;
}

__device__ __forceinline__ int warp_sum_i(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(FULL, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
    return v;
}

// q8 of one element given its group's absmax (the rule of colibri_q8_quantize).
__device__ __forceinline__ int q8_code(float x, float d)
{
    if (d == 0.0f)
        return 0;
    float v = roundf(__fdiv_rn(x, d));
    v = fminf(fmaxf(v, -127.0f), 127.0f);
    return (int)v;
}

// q8_code(x, d) given r = fp32(1/d) (__frcp_rn), the same code with one multiplication in
// place of the division, except next to a rounding boundary. With f = fp32(x/d) and
// y = fp32(x * r), |y - f| <= |x/d| * (2^-23 + 2^-24 + 2^-48) <= 2.3e-5 while |x/d| <= 128,
// so roundf(y) == roundf(f) whenever y is more than 1e-4 away from every half-integer;
// nearer (and for any y that is not a finite value below 128 in magnitude) the exact
// division decides.
__device__ __forceinline__ int q8_code_r(float x, float d, float r)
{
    if (d == 0.0f)
        return 0;
    const float y = x * r;
    float v;
    if (fabsf(y) <= 128.0f && fabsf(y - floorf(y) - 0.5f) > 1e-4f)
        v = roundf(y);
    else
        v = roundf(__fdiv_rn(x, d));
    v = fminf(fmaxf(v, -127.0f), 127.0f);
    return (int)v;
}

// ---- mbarrier + 1-D bulk copy (cp.async.bulk) ---------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Asynchronous global -> shared copies (no registers held while in flight): 16 or 4 bytes
// to dst, of which src_bytes (0 or the full size) come from src and the rest are zeros;
// src must be 16- (4-) byte aligned. Complete after cp_async_wait_all() by the issuing
// thread.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async4(void *dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// The thread's cp.async copies issued since the last commit form one group.
__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most N of the thread's committed groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait_group()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

// Ends an mbarrier's life, so that its word may be initialised again.
__device__ __forceinline__ void mbar_inval(uint64_t *bar)
{
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Barrier among `threads` threads (a multiple of 32) of the CTA on hardware barrier `id`.
__device__ __forceinline__ void named_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(addr), "r"(parity), "r"(WAIT_HINT_NS)
        : "memory");
    return done != 0;
}

// The rest of a wait that did not end at the first try (one copy of this code for all
// call sites): false after WAIT_LIMIT_NS.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t *bar, uint32_t parity)
{
    const uint32_t addr = smem_u32(bar);
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(addr, parity))
            return true;
        if (global_ns() - t0 > WAIT_LIMIT_NS)
            return false;
    }
}

// Returns true once the phase with the given parity has completed, false after
// WAIT_LIMIT_NS. Each try_wait suspends the thread (up to WAIT_HINT_NS) until the phase
// completes.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    return mbar_try_wait(smem_u32(bar), parity) || mbar_wait_slow(bar, parity);
}

// Hint: bring [src, src + bytes) into L2 (no completion to wait for). src 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// L2 policy for bytes read once per call: evicted first, so they do not push out lines
// that are still to be used (a prefetched shared expert, small tables).
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the kernel before it still runs; grid_dep_wait() blocks
// the calling thread until that kernel has completed and its writes are visible.
// grid_dep_launch() lets the dependent kernel be scheduled before this one ends.
__device__ __forceinline__ void grid_dep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_dep_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The key a router score is ranked by: the score, or -inf for NaN, so that the order
// (larger first, then lower index) is total and a selection always yields distinct,
// valid ids.
__device__ __forceinline__ float rank_score(float v)
{
    return v != v ? -INFINITY : v;
}

__device__ __forceinline__ int ld_acquire_gpu(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Waits until *p >= target (a counter other CTAs raise); false after WAIT_LIMIT_NS.
__device__ __forceinline__ bool wait_count_geq(const int *p, int target)
{
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (ld_acquire_gpu(p) >= target)
            return true;
        const uint64_t now = global_ns();
        if (i == 0)
            t0 = now;
        else if (now - t0 > WAIT_LIMIT_NS)
            return false;
        __nanosleep(64);
    }
}

// Global -> shared bulk copy; dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Per-slot work description written by the bucketing kernel.
struct Slot {
    int expert;  // routed expert id, or -1 for the shared expert
    int begin;   // first entry in the pair list (routed) / 0 (shared)
    int count;   // tokens routed to this slot
    int pad;
};

// Device counters written by the bucketing kernel.
struct Counters {
    int n_slots;
    int n_items_gateup;
    int n_items_down;
    int n_routed;
    int n_rows;  // rows of h and y: the pairs listed in slots + the shared expert's T
    int pad[3];
};

}  // namespace clb
