// qk_device.cuh -- device helpers shared by the library's kernels (sm_103a).
//
// Hand-written PTX for the asynchronous machinery: mbarriers, 1-D bulk copies
// global -> shared (cp.async.bulk), named barriers, and bounded waits.  Every
// wait is bounded by a wall-clock limit read from %globaltimer; a wait that
// runs out returns false and the caller records QK_ERR_TIMEOUT in the device
// error word and leaves the kernel.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace qk {

constexpr int kErrTimeout = 1;   // bits in the device error word: a bounded wait ran out,
constexpr int kErrBadIndex = 2;  // an index read from device memory was out of range

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// An arrival by the threads whose `pred` is true, without a branch.
__device__ __forceinline__ void mbar_arrive_if(uint32_t bar, bool pred)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}"
                 ::"r"(bar), "r"(static_cast<uint32_t>(pred)) : "memory");
}

// Announce `bytes` more transaction bytes for the current phase without an
// arrival (the phase still needs its expected arrivals).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
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

// The same test with a suspend-time hint: the thread may sleep (without
// taking issue slots) until the phase completes or about hint_ns pass.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Wait (sleeping between tests) until the phase with the given parity has
// completed, for at most limit_ns of wall-clock time.  Returns false if the
// limit ran out.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    const uint64_t deadline = globaltimer_ns() + limit_ns;
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (globaltimer_ns() > deadline) return false;
    }
}

// Wait until the phase with the given parity has completed, for at most
// limit_ns of wall-clock time.  Returns false if the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t deadline = globaltimer_ns() + limit_ns;
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 0 && globaltimer_ns() > deadline) return false;
    }
}

// ---------------------------------------------------------------- bulk copy

// L2 policy: the weights are streamed once, so they are marked evict-first
// to keep activations and outputs resident in L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy of `bytes` (multiple of 16) from global `src` (16-byte aligned)
// into shared `dst` (16-byte aligned); completion is signalled on `bar` as
// transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// ---------------------------------------------------------------- named barriers

__device__ __forceinline__ void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- numerics helpers

// fp16 bits -> fp32 (exact), through the CUDA half conversion.
__device__ __forceinline__ float half_bits_to_float(uint32_t h16)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h16 & 0xFFFFu)));
}

// SwiGLU's gate: silu(z) = z / (1 + e^-z), with CUDA's expf and its fast
// division (within 2 ulp of the correctly rounded quotient).  Gate sums of a
// few hundred are common, where e^-z overflows; the IEEE division by
// infinity leaves its fast path, at a cost that showed in whole kernels, so a
// denominator beyond the fast division's range (2^126) gives the limit, a
// zero of z's sign.
__device__ __forceinline__ float silu(float z)
{
    const float den = 1.0f + expf(-z);
    return den < 8.5e37f ? __fdividef(z, den) : 0.0f * z;
}

constexpr uint32_t kMagic = 0x4B000000u;   // 2^23 as an fp32 bit pattern
constexpr float kTwo23 = 8388608.0f;

// ---------------------------------------------------------------- packed fp32 pairs
// A float pair lives in one 64-bit register pair (low half = first value);
// the arithmetic is done with the f32x2 instructions.

// Magic float 2^23 + field: one LOP3 computing (w & mask) | 0x4B000000.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t magic_field(uint32_t w)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "n"(MASK), "n"(0x4B000000));
    return r;
}

__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}

__device__ __forceinline__ uint64_t pack2f(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float2 unpack2f(uint64_t v)
{
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// ---------------------------------------------------------------- 4-way byte dot products
// d = c + sum_{i<4} a.byte[i] * b.byte[i]; U/S = unsigned/signed bytes of a, b.
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// ---------------------------------------------------------------- sub-warp reductions
// redux.sync over the lanes named in `mask` (every lane of the mask executes
// the same instruction with the same mask; disjoint groups of a warp may
// reduce at once, each with its own mask).
__device__ __forceinline__ uint32_t redux_max_u32(uint32_t mask, uint32_t v)
{
    uint32_t r;
    asm volatile("redux.sync.max.u32 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(mask));
    return r;
}
__device__ __forceinline__ uint32_t redux_add_u32(uint32_t mask, uint32_t v)
{
    uint32_t r;
    asm volatile("redux.sync.add.u32 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(mask));
    return r;
}
__device__ __forceinline__ int redux_add_s32(uint32_t mask, int v)
{
    int r;
    asm volatile("redux.sync.add.s32 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(mask));
    return r;
}

__device__ __forceinline__ void record_error(int *err, int bit)
{
    if (err) atomicOr(err, bit);
}

}  // namespace qk
