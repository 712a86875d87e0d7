// tc_common.cuh -- inline-PTX building blocks of the sm_103a kernels: mbarriers with bounded
// waits, TMA tensor loads, bulk copies, tcgen05 (TMEM allocation, MMA, commit, loads) and the
// shared-memory matrix / instruction descriptors of tcgen05.mma.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include <atomic>
#include <type_traits>

#include "fcm_device.cuh"
#include "fcm_internal.h"

namespace fcm {
namespace tc {

// Index checks of a debug build (compiled with FCM_DEBUG_CHECKS; nothing in a release build).
// A failed check never traps: it sets FCM_DEVERR_CHECK in the device error word (err[0]) and
// records the first failure as (check id << 24) | (offending index & 0xFFFFFF) in err[1], which
// fcm_check reports; the access itself still happens, inside the buffer the check guards.
__device__ __forceinline__ void fcm_dcheck_fail(unsigned *err, unsigned id, unsigned idx) {
    atomicOr(err, 2u);   // FCM_DEVERR_CHECK
    atomicCAS(err + 1, 0u, (id << 24) | (idx & 0xFFFFFFu));
}
#ifdef FCM_DEBUG_CHECKS
#define FCM_DCHECK(cond, err, id, idx)                                                 \
    do {                                                                               \
        if (!(cond)) fcm::tc::fcm_dcheck_fail((err), (unsigned)(id), (unsigned)(idx)); \
    } while (0)
#else
#define FCM_DCHECK(cond, err, id, idx) \
    do {                                \
    } while (0)
#endif

// A wait gives up after this long (ns) and reports FCM_DEVERR_TIMEOUT.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------- programmatic dependent launch
// The kernels are launched with programmatic stream serialization allowed (launch_pdl below):
// a kernel may start while the previous kernel on the stream finishes, so its prologue (barrier
// set-up, TMEM allocation, copies of the handle's weights, which no kernel writes) overlaps that
// tail.  Before its first read of activations -- which a previous kernel may have written -- a
// kernel waits for the previous grid to complete and its memory to be visible (pdl_wait); every
// global write of the kernels depends on such a read.  Each CTA lets the next kernel start
// launching once its own prologue is done (pdl_launch_dependents).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Largest dynamic shared memory of a CTA on sm_103a.
constexpr int kSmemOptin = 227 * 1024;

// Launches a persistent kernel with programmatic stream serialization allowed.  The kernel's
// dynamic shared-memory limit is raised to kSmemOptin once per context (attr_ctx, one per kernel
// instantiation, holds the context it was raised in): a new context -- another device, or after
// a device reset -- raises it again.
template <typename A>
inline cudaError_t launch_pdl(void (*kernel)(A), std::atomic<unsigned long long> &attr_ctx,
                              int ctas, int threads, uint32_t smem, cudaStream_t st, const A &a) {
    if (smem > (uint32_t)kSmemOptin) return cudaErrorInvalidValue;
    const unsigned long long ctx = fcm_current_ctx_id();
    if (ctx == 0 || attr_ctx.load(std::memory_order_relaxed) != ctx) {
        const cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOptin);
        if (e != cudaSuccess) return e;
        attr_ctx.store(ctx, std::memory_order_relaxed);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// ------------------------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of parity `parity` to complete.  Gives up (returns false) when
// another warp already gave up (*abort != 0) or after `limit_ns`; in the latter case it sets
// FCM_DEVERR_TIMEOUT in the device error word and raises *abort for the whole CTA.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          unsigned *err, unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                atomicOr(err, 1u);  // FCM_DEVERR_TIMEOUT
                *abort = 1;
                return false;
            }
        }
    }
}

// 16-byte shared-memory load and store by 32-bit shared address.
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ void sts64(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared.v2.b32 [%0], {%1,%2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

// ----------------------------------------------------------------------------------- TMA
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *tmap, uint32_t bar, int c0,
                                            int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, uint32_t bar, int c0,
                                            int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

// 1-D bulk copy global -> shared (size and both addresses multiples of 16 bytes).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// Tensor stores shared -> global (bulk async-group completion; out-of-range box parts are
// clipped by the TMA unit).
__device__ __forceinline__ void tma_store_4d(const void *tmap, uint32_t src, int c0, int c1, int c2,
                                             int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::
            "l"(reinterpret_cast<uint64_t>(tmap)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ void tma_store_2d(const void *tmap, uint32_t src, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(tmap)),
        "r"(src), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed bulk groups are still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Barrier among `nthreads` threads (a multiple of 32) on hardware barrier `id` (1..15).
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier among `nthreads` threads on barrier `id` that also returns the OR of `pred` over
// them, so that every participant takes the same branch afterwards.
__device__ __forceinline__ bool named_barrier_or(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// ------------------------------------------------------- mixed-precision multiply-add
// acc0 += lo(x2) * lo(w2), acc1 += hi(x2) * hi(w2): 16-bit inputs, exact products, fp32 sum
// rounded once (the same result as widening both inputs to fp32 and using fmaf).
template <typename T> struct Fma16;
template <> struct Fma16<__half> {
    static __device__ __forceinline__ void fma2(float &acc0, float &acc1, uint32_t x2, uint32_t w2) {
        asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
            "mov.b32 {xl, xh}, %2;\n\tmov.b32 {wl, wh}, %3;\n\t"
            "fma.rn.f32.f16 %0, xl, wl, %0;\n\tfma.rn.f32.f16 %1, xh, wh, %1;\n\t}"
            : "+f"(acc0), "+f"(acc1)
            : "r"(x2), "r"(w2));
    }
};
template <> struct Fma16<__nv_bfloat16> {
    static __device__ __forceinline__ void fma2(float &acc0, float &acc1, uint32_t x2, uint32_t w2) {
        asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
            "mov.b32 {xl, xh}, %2;\n\tmov.b32 {wl, wh}, %3;\n\t"
            "fma.rn.f32.bf16 %0, xl, wl, %0;\n\tfma.rn.f32.bf16 %1, xh, wh, %1;\n\t}"
            : "+f"(acc0), "+f"(acc1)
            : "r"(x2), "r"(w2));
    }
};

// Round two fp32 values to a packed 16-bit pair (round to nearest even; `lo` in the low half)
// and apply activation ACT (0 none, 1 ReLU, 2 ReLU6): the conversion itself clamps at 0
// (cvt .relu), then ReLU6 takes the minimum with 6 on the pair.  Clamping after rounding
// equals rounding after clamping because rounding is monotonic and 0 and 6 are exact.  ACT is a
// template parameter so that the per-element code has no branches.
template <typename T> struct Pack2;
template <> struct Pack2<__half> {
    template <int ACT>
    static __device__ __forceinline__ uint32_t run(float lo, float hi) {
        uint32_t r;
        if (ACT == 0)
            asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        else
            asm("cvt.rn.relu.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        if (ACT == 2) {
            __half2 h = *reinterpret_cast<__half2 *>(&r);
            h = __hmin2(h, __float2half2_rn(6.0f));
            r = *reinterpret_cast<uint32_t *>(&h);
        }
        return r;
    }
};
template <> struct Pack2<__nv_bfloat16> {
    template <int ACT>
    static __device__ __forceinline__ uint32_t run(float lo, float hi) {
        uint32_t r;
        if (ACT == 0)
            asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        else
            asm("cvt.rn.relu.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        if (ACT == 2) {
            __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&r);
            h = __hmin2(h, __float2bfloat162_rn(6.0f));
            r = *reinterpret_cast<uint32_t *>(&h);
        }
        return r;
    }
};

// ------------------------------------------------------- INT8 storage
// int8 values are exact in f16 and the products of two of them exact in fp32, so the INT8
// module runs on the 16-bit paths: the tensor core multiplies f16 images of int8 operands into
// an fp32 accumulator (exact while every partial sum stays below 2^22), and the depthwise
// stencil uses the mixed-precision f16 FMA.
struct I8 {
    // Offset carried by widened inputs: 1024 (the f16 pattern 0x6400, whose ulp is 1) + 128.
    static constexpr float kBias = 1152.0f;
    // Four int8 lanes -> two f16x2 holding 1152 + x: the byte x ^ 0x80 = x + 128 (0..255) is
    // placed in the low mantissa bits of 0x6400.  The stencil sums (1152 + x) * w over its taps
    // starting from -1152 * (sum of the channel's taps); every step is exact.
    static __device__ __forceinline__ void widen4(uint32_t x4, uint32_t &lo, uint32_t &hi) {
        const uint32_t u = x4 ^ 0x80808080u;
        lo = __byte_perm(u, 0x64646464u, 0x4140);
        hi = __byte_perm(u, 0x64646464u, 0x4342);
    }
    // Requantization of v = s * acc + b: clamp to the activation's integer range (none
    // [-128, 127], ReLU [0, 127], ReLU6 [0, 6]; clamping to integer bounds commutes with
    // rounding), then round to the nearest integer, ties to even, by adding 1.5 * 2^23 (ulp 1
    // there): the sum holds the integer r, and its low byte is r as an int8.
    static constexpr float kRound = 12582912.0f;
    template <int ACT>
    static __device__ __forceinline__ float biased(float v) {
        const float lo = ACT == 0 ? -128.0f : 0.0f;
        const float hi = ACT == 2 ? 6.0f : 127.0f;
        return __fadd_rn(fminf(fmaxf(v, lo), hi), kRound);
    }
    // Two requantized values as f16x2 (`lo` in the low half): the A operand of the 1x1 GEMM.
    // With ReLU/ReLU6 the lower clamp is the conversion's own .relu: any negative v rounds to
    // a value <= 0 (rounding is monotonic), which .relu turns into 0.
    template <int ACT>
    static __device__ __forceinline__ uint32_t half2(float lo, float hi) {
        uint32_t r;
        if (ACT == 0) {
            const float rl = __fsub_rn(biased<ACT>(lo), kRound);
            const float rh = __fsub_rn(biased<ACT>(hi), kRound);
            asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(rh), "f"(rl));
        } else {
            const float top = ACT == 2 ? 6.0f : 127.0f;
            const float rl = __fsub_rn(__fadd_rn(fminf(lo, top), kRound), kRound);
            const float rh = __fsub_rn(__fadd_rn(fminf(hi, top), kRound), kRound);
            asm("cvt.rn.relu.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(rh), "f"(rl));
        }
        return r;
    }
    // Four requantized values packed as int8 lanes (a in the lowest byte).
    template <int ACT>
    static __device__ __forceinline__ uint32_t bytes4(float a, float b, float c, float d) {
        const uint32_t ta = __float_as_uint(biased<ACT>(a)), tb = __float_as_uint(biased<ACT>(b));
        const uint32_t tc = __float_as_uint(biased<ACT>(c)), td = __float_as_uint(biased<ACT>(d));
        return __byte_perm(__byte_perm(ta, tb, 0x0040), __byte_perm(tc, td, 0x0040), 0x5410);
    }
};

// Calls f(std::integral_constant<int, act>{}) for a runtime activation code 0, 1 or 2, so that a
// role's loop is compiled once per activation.
template <typename F>
__device__ __forceinline__ void with_act(int act, F &&f) {
    if (act == 0)
        f(std::integral_constant<int, 0>{});
    else if (act == 1)
        f(std::integral_constant<int, 1>{});
    else
        f(std::integral_constant<int, 2>{});
}

// -------------------------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
                 "r"(ncols)
                 : "memory");
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

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (fp16 or bf16 inputs, fp32 accumulator).
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp gets TMEM lane
// (warp's quarter * 32 + i), columns col .. col+15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// The same wait with the registers of two 16-column loads tied to it: the registers a
// tcgen05.ld writes are valid only after the wait, and the ties keep the compiler from
// scheduling any use of them before it (the second array may be unused by the caller).
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&a)[16], uint32_t (&b)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]),
                   "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]),
                   "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(b[0]), "+r"(b[1]),
                   "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]),
                   "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]),
                   "+r"(b[14]), "+r"(b[15])
                 :
                 : "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzled canonical
// layout: 8-row x 128-byte atoms (row r's 16-byte chunk c stored at chunk c ^ (r & 7)),
// consecutive 8-row groups 1024 bytes apart.  Atoms must start on 1024-byte boundaries.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);      // start address
    d |= (uint64_t)1 << 16;                        // leading byte offset (unused here)
    d |= (uint64_t)(1024u >> 4) << 32;             // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;                        // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                        // 128-byte swizzle
    return d;
}

// The descriptor of the operand `bytes` further on (a multiple of 16): the start-address field
// holds address / 16 in 14 bits and shared memory ends below 2^18 bytes, so the field never
// carries into the next one.
__device__ __forceinline__ uint64_t desc_advance(uint64_t d, uint32_t bytes) {
    return d + (uint64_t)(bytes >> 4);
}

// Byte offset of the 16-wide K step k16 in a K-major operand of `rows` rows stored as 64-wide
// K blocks of 128-byte swizzled rows.
__device__ __forceinline__ uint32_t k16_offset(int k16, int rows) {
    return (uint32_t)(k16 >> 2) * (uint32_t)rows * 128u + (uint32_t)(k16 & 3) * 32u;
}

// Instruction descriptor of kind::f16 with fp32 accumulation, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int m, int n) {
    return (1u << 4)                              // D format: f32
           | ((bf16 ? 1u : 0u) << 7)              // A format: f16 / bf16
           | ((bf16 ? 1u : 0u) << 10)             // B format
           | ((uint32_t)(n >> 3) << 17)           // N / 8
           | ((uint32_t)(m >> 4) << 24);          // M / 16
}

// Byte offset of element (row, k) of a K-major operand with `rows` rows stored as 64-wide
// K blocks of 128-byte swizzled rows (block kb holds k in [64kb, 64kb+64)).
__host__ __device__ inline uint32_t sw128_offset(int row, int k, int rows, int esize) {
    int kb = k / 64;
    int chunk = ((k % 64) * esize) / 16;
    int within = ((k % 64) * esize) % 16;
    return (uint32_t)(kb * rows * 128 + row * 128 + ((chunk ^ (row & 7)) << 4) + within);
}

}  // namespace tc
}  // namespace fcm
