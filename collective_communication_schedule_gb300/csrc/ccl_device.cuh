// Device helpers shared by the executor kernels: gpu-scope flag access,
// bounded waits, and the 16-byte vector copy / reduce bodies.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "ccl_executor.cuh"

namespace ccl {

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(unsigned long long* p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed(unsigned long long* p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// acquire-release fence at gpu scope: after relaxed loads that observed a
// flag it acts as the acquire; before relaxed flag stores, as the release
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ unsigned long long gtimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait by one thread: returns false when the limit passes or
// another threadblock has already failed (status[0] != 0).  On timeout the
// first failing threadblock records (code, block, step, reason) in status.
__device__ __forceinline__ bool wait_geq(const unsigned long long* p, unsigned long long v, int* status,
                                         unsigned long long timeout_ns, int si, int reason,
                                         unsigned long long& waited)
{
    if (ld_acquire(p) >= v) return true;
    unsigned long long t0 = gtimer();
    unsigned spins = 0;
    while (true) {
        if (ld_acquire(p) >= v) break;
        ++spins;
        if ((spins & 15) == 0) {
            if (*(volatile int*)status != 0) return false;
            unsigned long long now = gtimer();
            if (now - t0 > timeout_ns) {
                if (atomicCAS(status, 0, (int)CCL_ERR_TIMEOUT) == 0) {
                    status[1] = blockIdx.x;
                    status[2] = si;
                    status[3] = reason;
                }
                return false;
            }
        }
        if (spins > 64) __nanosleep(64);
    }
    waited += gtimer() - t0;
    return true;
}

template <int DT>
__device__ __forceinline__ uint32_t add2(uint32_t a, uint32_t b);

template <>
__device__ __forceinline__ uint32_t add2<CCL_F32>(uint32_t a, uint32_t b)
{
    return __float_as_uint(__uint_as_float(a) + __uint_as_float(b));
}
template <>
__device__ __forceinline__ uint32_t add2<CCL_I32>(uint32_t a, uint32_t b)
{
    return a + b;  // modulo 2^32
}
template <>
__device__ __forceinline__ uint32_t add2<CCL_BF16>(uint32_t a, uint32_t b)
{
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
    __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
    float2 fx = __bfloat1622float2(x), fy = __bfloat1622float2(y);
    __nv_bfloat162 r = __floats2bfloat162_rn(fx.x + fy.x, fx.y + fy.y);
    return *reinterpret_cast<uint32_t*>(&r);
}
template <>
__device__ __forceinline__ uint32_t add2<CCL_F16>(uint32_t a, uint32_t b)
{
    __half2 x = *reinterpret_cast<__half2*>(&a);
    __half2 y = *reinterpret_cast<__half2*>(&b);
    float2 fx = __half22float2(x), fy = __half22float2(y);
    __half2 r = __floats2half2_rn(fx.x + fy.x, fx.y + fy.y);
    return *reinterpret_cast<uint32_t*>(&r);
}

template <int DT>
__device__ __forceinline__ uint4 vadd(uint4 a, uint4 b)
{
    return make_uint4(add2<DT>(a.x, b.x), add2<DT>(a.y, b.y), add2<DT>(a.z, b.z), add2<DT>(a.w, b.w));
}

__device__ __forceinline__ uint4 vload(const uint4* p, bool stream) { return stream ? __ldcs(p) : __ldcg(p); }
__device__ __forceinline__ void vstore(uint4* p, uint4 v, bool stream)
{
    if (stream) __stcs(p, v); else __stcg(p, v);
}

// 16-byte path: nv vectors; full tiles keep U vectors per operand in flight
// per thread, the remainder goes one vector per thread.
template <bool RED, int DT>
__device__ __forceinline__ void move_vec(const uint4* a, bool as, const uint4* b, bool bs, uint4* o1, bool o1s,
                                         uint4* o2, int64_t nv, int tid, int T)
{
    constexpr int U = 4;   // vectors in flight per operand per thread
    int64_t i = tid;
    const int64_t full = nv - (int64_t)(U - 1) * T;
    for (; i < full; i += (int64_t)U * T) {
        uint4 va[U], vb[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            va[u] = vload(a + i + u * T, as);
            if (RED) vb[u] = vload(b + i + u * T, bs);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            uint4 r = va[u];
            if (RED) r = vadd<DT>(va[u], vb[u]);
            vstore(o1 + i + u * T, r, o1s);
            if (o2) vstore(o2 + i + u * T, r, false);
        }
    }
    // what is left of this thread's vectors (at most U - 1) in one round:
    // all of its loads in flight together instead of one round trip each
    // (loads past the end re-read the last vector and are not used)
    if (i < nv) {
        uint4 va[U - 1], vb[U - 1];
#pragma unroll
        for (int u = 0; u < U - 1; ++u) {
            const int64_t j = i + u * T < nv ? i + u * T : nv - 1;
            va[u] = vload(a + j, as);
            if (RED) vb[u] = vload(b + j, bs);
        }
#pragma unroll
        for (int u = 0; u < U - 1; ++u)
            if (i + u * T < nv) {
                uint4 r = va[u];
                if (RED) r = vadd<DT>(va[u], vb[u]);
                vstore(o1 + i + u * T, r, o1s);
                if (o2) vstore(o2 + i + u * T, r, false);
            }
    }
}

// element path (unaligned operands or the tail of a piece)
template <bool RED, int DT>
__device__ void move_elem(const char* a, const char* b, char* o1, char* o2, int64_t lo, int64_t hi, int tid, int T)
{
    constexpr int ES = (DT == CCL_BF16 || DT == CCL_F16) ? 2 : 4;
    for (int64_t i = lo + tid; i < hi; i += T) {
        if (ES == 4) {
            uint32_t x = __ldcg(reinterpret_cast<const unsigned int*>(a) + i);
            if (RED) x = add2<DT>(x, __ldcg(reinterpret_cast<const unsigned int*>(b) + i));
            if (o1) __stcg(reinterpret_cast<unsigned int*>(o1) + i, x);
            if (o2) __stcg(reinterpret_cast<unsigned int*>(o2) + i, x);
        } else {
            uint32_t x = __ldcg(reinterpret_cast<const unsigned short*>(a) + i);
            if (RED) {
                uint32_t y = __ldcg(reinterpret_cast<const unsigned short*>(b) + i);
                x = add2<DT>(x, y) & 0xffffu;  // low half holds the element
            }
            if (o1) __stcg(reinterpret_cast<unsigned short*>(o1) + i, (unsigned short)x);
            if (o2) __stcg(reinterpret_cast<unsigned short*>(o2) + i, (unsigned short)x);
        }
    }
}

template <bool RED, int DT>
__device__ __forceinline__ void move(const char* a, bool as, const char* b, bool bs, char* o1, bool o1s, char* o2,
                                     int64_t n, int tid, int T)
{
    constexpr int ES = (DT == CCL_BF16 || DT == CCL_F16) ? 2 : 4;
    constexpr int VE = 16 / ES;
    uintptr_t al = (uintptr_t)a | (uintptr_t)o1 | (uintptr_t)o2 | (RED ? (uintptr_t)b : 0);
    int64_t nv = 0;
    if ((al & 15) == 0) {
        nv = n / VE;
        move_vec<RED, DT>(reinterpret_cast<const uint4*>(a), as, reinterpret_cast<const uint4*>(b), bs,
                          reinterpret_cast<uint4*>(o1), o1s, reinterpret_cast<uint4*>(o2), nv, tid, T);
    }
    if (nv * VE < n) move_elem<RED, DT>(a, b, o1, o2, nv * VE, n, tid, T);
}

// copy or reduce n elements, shared by threads [0, T) of the caller (tid)
template <int DT>
__device__ __forceinline__ void move_part(bool red, const char* a, bool as, const char* b, bool bs, char* o1,
                                          bool o1s, char* o2, int64_t n, int tid, int T)
{
    if (red) move<true, DT>(a, as, b, bs, o1, o1s, o2, n, tid, T);
    else move<false, DT>(a, as, b, bs, o1, o1s, o2, n, tid, T);
}

// the whole CTA moves the data
template <int DT>
__device__ __forceinline__ void move_dt(bool red, const char* a, bool as, const char* b, bool bs, char* o1,
                                        bool o1s, char* o2, int64_t n)
{
    move_part<DT>(red, a, as, b, bs, o1, o1s, o2, n, threadIdx.x, blockDim.x);
}

// ---------------------------------------------------------------- LL lines
// An LL line is one 64-bit word: 4 data bytes in the low half, the flag of
// its FIFO slot (sequence number + 1, low 32 bits) in the high half.  Lines
// are written and read as elements of 16-byte vectors; each 64-bit element
// is an aligned scalar access and therefore single-copy atomic, so a reader
// that sees the flag sees the data beside it.  Volatile accesses bypass L1.
__device__ __forceinline__ void ll_load2(const void* p, unsigned long long& x, unsigned long long& y)
{
    asm volatile("ld.volatile.global.v2.u64 {%0, %1}, [%2];" : "=l"(x), "=l"(y) : "l"(p) : "memory");
}
__device__ __forceinline__ void ll_store2(void* p, unsigned long long x, unsigned long long y)
{
    asm volatile("st.volatile.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(x), "l"(y) : "memory");
}
__device__ __forceinline__ unsigned long long ll_line(unsigned data, unsigned flag)
{
    return ((unsigned long long)flag << 32) | data;
}
// the 16 data bytes of vector i as four lines (32 bytes) at p + 32 i
__device__ __forceinline__ void ll_store_vec(char* p, long long i, uint4 r, unsigned flag)
{
    char* q = p + 32 * i;
    ll_store2(q, ll_line(r.x, flag), ll_line(r.y, flag));
    ll_store2(q + 16, ll_line(r.z, flag), ll_line(r.w, flag));
}

// ---------------------------------------------------------------- mbarriers
__device__ __forceinline__ unsigned smem_addr(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(unsigned long long* bar, int count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// arrive (release at CTA scope)
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
                 : "memory");
}

// arrive and add `bytes` to the transaction count the phase waits for
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, unsigned bytes)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// ------------------------------------------------------- bulk (TMA) copies
// global -> shared, completion counted on an mbarrier (16-byte aligned, size
// a multiple of 16)
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, unsigned bytes, unsigned long long* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(smem_dst)),
                 "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}
// shared -> global, tracked by the issuing thread's bulk groups
__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, unsigned bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_addr(smem_src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most n (clamped to 7) of this thread's bulk groups are still
// reading shared memory / still pending
__device__ __forceinline__ void bulk_wait_read(int n)
{
    switch (n < 0 ? 0 : (n > 7 ? 7 : n)) {
    case 0: asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.bulk.wait_group.read 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.bulk.wait_group.read 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.bulk.wait_group.read 6;" ::: "memory"); break;
    default: asm volatile("cp.async.bulk.wait_group.read 7;" ::: "memory"); break;
    }
}
__device__ __forceinline__ void bulk_wait(int n)
{
    switch (n < 0 ? 0 : (n > 7 ? 7 : n)) {
    case 0: asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.bulk.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.bulk.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.bulk.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.bulk.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.bulk.wait_group 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.bulk.wait_group 6;" ::: "memory"); break;
    default: asm volatile("cp.async.bulk.wait_group 7;" ::: "memory"); break;
    }
}
// order generic-proxy and async-proxy accesses (global memory / this CTA's
// shared memory)
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// test of the phase with the given parity that may suspend the thread for a
// short, hardware-chosen time while the phase is incomplete (acquire at CTA
// scope); false when the phase has not completed yet
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, unsigned parity)
{
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// non-blocking test of the phase with the given parity (acquire at CTA scope)
__device__ __forceinline__ bool mbar_test(unsigned long long* bar, unsigned parity)
{
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

}  // namespace ccl
