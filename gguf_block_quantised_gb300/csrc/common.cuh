// common.cuh -- device helpers shared by the libqmv kernels (sm_103a).
//
// Inline PTX for the Blackwell data movers (mbarrier, cp.async.bulk), integer
// dot products (dp4a) and a bounded-wait discipline: every spin on an
// mbarrier gives up after a time limit, records a fault in the device status
// word and lets the kernel return, so a stuck copy can never hang the GPU.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/qmv.h"

// Device status word bits (read and cleared by qmv_get_status).
#define QMV_DEV_BAD_EXPERT 1u
#define QMV_DEV_WAIT_TIMEOUT 2u
#define QMV_DEV_BAD_ARG 4u

#define QMV_WAIT_LIMIT_NS 2000000000ull   // 2 s: a copy that has not landed by then never will

namespace qmv {

// Format traits that kernels, launchers and the boundary share.
__host__ __device__ constexpr bool kq_rt(int T)   // 256-element K-quant (Q8_K activations)
{
    return T == QMV_Q4_K || T == QMV_Q6_K || T == QMV_Q5_K || T == QMV_Q2_K || T == QMV_Q3_K;
}
__host__ __device__ constexpr bool plain_rt(int T) { return T == QMV_F32 || T == QMV_F16 || T == QMV_BF16; }
// Run length of the fp32 activation sums the fp32-activation path stages for
// a format whose weights carry an offset (min) per run: 0 = none.
__host__ __device__ constexpr int xsum_run_rt(int T)
{
    return (T == QMV_Q4_K || T == QMV_Q5_K || T == QMV_Q4_1 || T == QMV_Q5_1) ? 32 : T == QMV_Q2_K ? 16 : 0;
}
__host__ __device__ constexpr int block_elems_rt(int T) { return kq_rt(T) ? 256 : plain_rt(T) ? 8 : 32; }

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier ---------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits with a limit under this many nanoseconds (set for diagnostics by
// qmv_set_wait_limit) poll without blocking and check the clock after every
// poll, so that they give up even when the phase completes a moment later.
constexpr uint64_t kShortWaitNs = 1000000ull;

__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

static __device__ __noinline__ bool mbar_wait_short(uint64_t* bar, uint32_t parity, unsigned* status, uint64_t limit_ns)
{
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_test_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(status, QMV_DEV_WAIT_TIMEOUT);
            return false;
        }
    }
}

// Wait for phase `parity` of `bar` to complete; false (and the status word
// flagged) if it has not after limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned* status,
                                                  uint64_t limit_ns = QMV_WAIT_LIMIT_NS)
{
    if (limit_ns < kShortWaitNs) return mbar_wait_short(bar, parity, status, limit_ns);
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(status, QMV_DEV_WAIT_TIMEOUT);
            return false;
        }
    }
}

// mbar_wait_bounded for warps off the critical path (producers that run ahead,
// an epilogue waiting a whole tile): between polls the warp sleeps for about
// sleep_ns, so that its polling does not take issue slots from the warps that
// do the work.
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t* bar, uint32_t parity, unsigned* status,
                                                  unsigned sleep_ns, uint64_t limit_ns = QMV_WAIT_LIMIT_NS)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        __nanosleep(sleep_ns);
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(status, QMV_DEV_WAIT_TIMEOUT);
            return false;
        }
    }
}

// ---- thread-block clusters: distributed shared memory and the barrier --------
// The address of this shared-memory location in the CTA of the cluster with
// rank `rank` (the same offset in its shared memory).
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank)
{
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    return a;
}

__device__ __forceinline__ void dsmem_st_u32(uint32_t a, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// All threads of all CTAs of the cluster; the stores before it (also into
// other CTAs' shared memory) are visible to every thread of the cluster after.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- bulk copy global -> shared (TMA, 1-D) ------------------------------------
// dst and src 16-byte aligned, bytes a multiple of 16.  Completion is signalled
// as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Hint the L2 to start fetching [src, src+bytes) (16-byte aligned, multiple of 16).
// Pull the 128-byte lines of [p, p + bytes) into L2, the lanes of one warp
// taking lines in turn.  A hint only: nothing returns to the thread, and a
// store by another grid to those lines still lands in L2, so it may precede
// the wait for the grid that writes them.
__device__ __forceinline__ void prefetch_l2_lines(const void* p, size_t bytes, int lane)
{
    if (bytes == 0) return;
    const char* c = static_cast<const char*>(p);
    const size_t n = bytes / 128 + 2;   // lines touched by an unaligned range
    for (size_t k = lane; k < n; k += 32) {
        const char* a = c + (k * 128 < bytes ? k * 128 : bytes - 1);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
    }
}

__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---- integer dot products ---------------------------------------------------------
// Four unsigned bytes of a times four signed bytes of b, plus c.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// Four signed bytes times four signed bytes, plus c.
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// ---- byte-addressed reads of shared memory -------------------------------------------
// K little-endian 32-bit words starting at any byte address p (shared memory,
// with at least 4 readable bytes after the last word's end).
template <int K>
__device__ __forceinline__ void load_words(const uint8_t* p, uint32_t (&w)[K])
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* base = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    const uint32_t sh = static_cast<uint32_t>(a & 3) * 8u;
    uint32_t prev = base[0];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const uint32_t next = base[k + 1];
        w[k] = __funnelshift_r(prev, next, sh);
        prev = next;
    }
}

__device__ __forceinline__ float half_bits_to_float(uint32_t h16)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h16 & 0xffffu)));
}

__device__ __forceinline__ uint32_t ld_u16(const uint8_t* p)   // 2-byte aligned
{
    return *reinterpret_cast<const uint16_t*>(p);
}

// Four unsigned bytes of w -> the float value of byte k minus `off`, exactly:
// 0x4B0000xx is the float 2^23 + xx, and 2^23 + off is exact below 2^24.
__device__ __forceinline__ float ubyte_to_float_minus(uint32_t w, int k, float two23_plus_off)
{
    return __int_as_float(static_cast<int>(__byte_perm(w, 0x4B000000u, 0x7650u + k))) - two23_plus_off;
}

// ---- the 8-bit activation quantiser step (shared by the quantise kernels and
// the matvec kernels that quantise their activations while staging them) ----
// d = amax/127 and id = 1/d (0 when d = 0), each one IEEE fp32 rounding.
__device__ __forceinline__ void act_scale(float amax, float& d, float& id)
{
    d = __fdiv_rn(amax, 127.f);
    id = d == 0.f ? 0.f : __fdiv_rn(1.f, d);
}
// q = round-half-away-from-zero(v * id), clamped to +-127.
__device__ __forceinline__ int8_t quant1(float v, float id)
{
    float r = roundf(__fmul_rn(v, id));
    r = fminf(fmaxf(r, -127.f), 127.f);
    return (int8_t)(int)r;
}

// A scale below 2^-128 (a block whose largest magnitude is under 127 * 2^-128)
// makes id = 1/d overflow, and v * id is then not the scaled value (0 * inf is
// not even a number).  Such a block's codes are round(v / d): the rare block
// divides its values by d first (one IEEE division each) and takes id = 1, so
// that quant1 multiplies by 1 exactly.  The common path computes no division
// (the loops are unrolled so that the arrays stay in registers).
template <int N>
__device__ __forceinline__ void tiny_scale_divide(float (&v)[N], float d, float& id)
{
    if (isinf(id)) {
#pragma unroll
        for (int k = 0; k < N; ++k) v[k] = __fdiv_rn(v[k], d);
        id = 1.f;
    }
}
template <int N>
__device__ __forceinline__ void tiny_scale_divide(float4 (&v)[N], float d, float& id)
{
    if (isinf(id)) {
#pragma unroll
        for (int k = 0; k < N; ++k)
            v[k] = make_float4(__fdiv_rn(v[k].x, d), __fdiv_rn(v[k].y, d), __fdiv_rn(v[k].z, d),
                               __fdiv_rn(v[k].w, d));
        id = 1.f;
    }
}

// ---- programmatic dependent launch ----------------------------------------------
// Wait until the grids this one depends on have finished and their writes are
// visible (a no-op when the kernel was not launched as a dependent).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next grid on the stream be scheduled (its own pdl_wait still waits
// for this grid to finish).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_sum_int(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---- MXFP8 activations (OCP Microscaling v1.0) -----------------------------------
// The scale exponent E of a 32-element block with largest magnitude amax:
// floor(log2(amax)) - 8 (8: the largest E4M3 exponent), at least -127; -127 for
// a block of zeros.  Stored as the E8M0 byte E + 127.
__device__ __forceinline__ int mx_scale_exp(float amax)
{
    const uint32_t b = __float_as_uint(amax);
    const int ef = (int)((b >> 23) & 0xffu);
    int lg;
    if (ef) lg = ef - 127;
    else if (b) lg = (31 - __clz((int)(b & 0x7fffffu))) - 149;   // subnormal amax
    else return -127;
    const int E = lg - 8;
    return E < -127 ? -127 : E;
}

// E4M3 code of x / 2^E: the scaling by a power of two is exact (a result
// below 2^-126 is far below half the smallest E4M3 step, so its rounding does
// not matter), then round to nearest even, magnitudes clamped to 448.
__device__ __forceinline__ uint32_t mx_e4m3(float x, int E)
{
    const float s = __uint_as_float((uint32_t)(127 - E) << 23);   // 2^-E, E in [-127, 119]
    return (uint32_t)__nv_cvt_float_to_fp8(__fmul_rn(x, s), __NV_SATFINITE, __NV_E4M3);
}

}  // namespace qmv
