// Device code shared by the executor kernels built with the library and the
// kernels generated for single plans at run time: gpu-scope flag access,
// bounded waits, the 16-byte vector copy / reduce bodies, LL lines,
// mbarriers and bulk copies.  It includes nothing but the layout header, so
// the run-time compiler (which has no standard headers) takes it as it is;
// element conversions are the hardware's round-to-nearest-even cvt
// instructions.
//
// The executor runs one CTA per threadblock program.  Per FIFO slot a step
// waits (bounded) until the incoming slot is full and the outgoing slot is
// free, the data path moves the slot's data with 16-byte accesses, and the
// flags are posted after a gpu-scope release fence.  The flag protocol
// stands in for the inter-GPU links of the pages' runtimes (MSCCLang report,
// §III.1 runtime; ReSCCL report, §II.2 kernel generation).
#pragma once

#include "ccl_layout.h"

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
// post a flag or counter: a release store when it is the only word posted
// (`alone`), else a relaxed store after the caller's fence
__device__ __forceinline__ void post_word(unsigned long long* p, unsigned long long v, bool alone)
{
    if (alone) st_release(p, v);
    else st_relaxed(p, v);
}
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
__device__ __forceinline__ unsigned add2(unsigned a, unsigned b);

template <>
__device__ __forceinline__ unsigned add2<CCL_F32>(unsigned a, unsigned b)
{
    return __float_as_uint(__uint_as_float(a) + __uint_as_float(b));
}
template <>
__device__ __forceinline__ unsigned add2<CCL_I32>(unsigned a, unsigned b)
{
    return a + b;  // modulo 2^32
}
// two packed bf16 / f16 elements: widen both to f32 exactly, add in f32,
// round the pair back to nearest even (low element in the low half)
template <>
__device__ __forceinline__ unsigned add2<CCL_BF16>(unsigned a, unsigned b)
{
    const float lo = __uint_as_float(a << 16) + __uint_as_float(b << 16);
    const float hi = __uint_as_float(a & 0xffff0000u) + __uint_as_float(b & 0xffff0000u);
    unsigned r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ void f16x2_to_f32(unsigned a, float& lo, float& hi)
{
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(a));
}
template <>
__device__ __forceinline__ unsigned add2<CCL_F16>(unsigned a, unsigned b)
{
    float xl, xh, yl, yh;
    f16x2_to_f32(a, xl, xh);
    f16x2_to_f32(b, yl, yh);
    unsigned r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(xh + yh), "f"(xl + yl));
    return r;
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
// per thread (4 in kernels built for 1024 threads, whose 64 registers a
// thread allows no more; 8 in kernels built for at most 512 threads), the
// remainder goes in one round.
template <bool RED, int DT, int U>
__device__ __forceinline__ void move_vec(const uint4* a, bool as, const uint4* b, bool bs, uint4* o1, bool o1s,
                                         uint4* o2, long long nv, int tid, int T)
{
    long long i = tid;
    const long long full = nv - (long long)(U - 1) * T;
    for (; i < full; i += (long long)U * T) {
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
            const long long j = i + u * T < nv ? i + u * T : nv - 1;
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
static __device__ void move_elem(const char* a, const char* b, char* o1, char* o2, long long lo, long long hi, int tid, int T)
{
    constexpr int ES = (DT == CCL_BF16 || DT == CCL_F16) ? 2 : 4;
    for (long long i = lo + tid; i < hi; i += T) {
        if (ES == 4) {
            unsigned x = __ldcg(reinterpret_cast<const unsigned int*>(a) + i);
            if (RED) x = add2<DT>(x, __ldcg(reinterpret_cast<const unsigned int*>(b) + i));
            if (o1) __stcg(reinterpret_cast<unsigned int*>(o1) + i, x);
            if (o2) __stcg(reinterpret_cast<unsigned int*>(o2) + i, x);
        } else {
            unsigned x = __ldcg(reinterpret_cast<const unsigned short*>(a) + i);
            if (RED) {
                unsigned y = __ldcg(reinterpret_cast<const unsigned short*>(b) + i);
                x = add2<DT>(x, y) & 0xffffu;  // low half holds the element
            }
            if (o1) __stcg(reinterpret_cast<unsigned short*>(o1) + i, (unsigned short)x);
            if (o2) __stcg(reinterpret_cast<unsigned short*>(o2) + i, (unsigned short)x);
        }
    }
}

// The data path is inlined into its callers; a translation unit may define
// CCL_MOVE_ATTR (e.g. __noinline__) first to keep one out-of-line copy.
#ifndef CCL_MOVE_ATTR
#define CCL_MOVE_ATTR __forceinline__
#endif

template <bool RED, int DT, int U>
__device__ CCL_MOVE_ATTR void move(const char* a, bool as, const char* b, bool bs, char* o1, bool o1s, char* o2,
                                     long long n, int tid, int T)
{
    constexpr int ES = (DT == CCL_BF16 || DT == CCL_F16) ? 2 : 4;
    constexpr int VE = 16 / ES;
    unsigned long long al = (unsigned long long)a | (unsigned long long)o1 | (unsigned long long)o2 | (RED ? (unsigned long long)b : 0);
    long long nv = 0;
    if ((al & 15) == 0) {
        nv = n / VE;
        move_vec<RED, DT, U>(reinterpret_cast<const uint4*>(a), as, reinterpret_cast<const uint4*>(b), bs,
                             reinterpret_cast<uint4*>(o1), o1s, reinterpret_cast<uint4*>(o2), nv, tid, T);
    }
    if (nv * VE < n) move_elem<RED, DT>(a, b, o1, o2, nv * VE, n, tid, T);
}

// copy or reduce n elements, shared by threads [0, T) of the caller (tid)
template <int DT, int U = 4>
__device__ __forceinline__ void move_part(bool red, const char* a, bool as, const char* b, bool bs, char* o1,
                                          bool o1s, char* o2, long long n, int tid, int T)
{
    if (red) move<true, DT, U>(a, as, b, bs, o1, o1s, o2, n, tid, T);
    else move<false, DT, U>(a, as, b, bs, o1, o1s, o2, n, tid, T);
}

// Three operands (a step that also takes the next step of a reduction chain:
// its local operand c is added after a + b, each sum rounded to the element
// type, as the two steps would).  Three quarters of the two-operand path's
// vectors in flight per operand (the registers of three operands).
template <int DT, int U>
__device__ __forceinline__ void move_vec3(const uint4* a, bool as, const uint4* b, bool bs, const uint4* c, bool cs,
                                          uint4* o1, bool o1s, uint4* o2, long long nv, int tid, int T)
{
    long long i = tid;
    const long long full = nv - (long long)(U - 1) * T;
    for (; i < full; i += (long long)U * T) {
        uint4 va[U], vb[U], vc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            va[u] = vload(a + i + u * T, as);
            vb[u] = vload(b + i + u * T, bs);
            vc[u] = vload(c + i + u * T, cs);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint4 r = vadd<DT>(vadd<DT>(va[u], vb[u]), vc[u]);
            vstore(o1 + i + u * T, r, o1s);
            if (o2) vstore(o2 + i + u * T, r, false);
        }
    }
    if (i < nv) {
        uint4 va[U - 1], vb[U - 1], vc[U - 1];
#pragma unroll
        for (int u = 0; u < U - 1; ++u) {
            const long long j = i + u * T < nv ? i + u * T : nv - 1;
            va[u] = vload(a + j, as);
            vb[u] = vload(b + j, bs);
            vc[u] = vload(c + j, cs);
        }
#pragma unroll
        for (int u = 0; u < U - 1; ++u)
            if (i + u * T < nv) {
                const uint4 r = vadd<DT>(vadd<DT>(va[u], vb[u]), vc[u]);
                vstore(o1 + i + u * T, r, o1s);
                if (o2) vstore(o2 + i + u * T, r, false);
            }
    }
}

template <int DT>
static __device__ void move_elem3(const char* a, const char* b, const char* c, char* o1, char* o2, long long lo,
                                  long long hi, int tid, int T)
{
    constexpr int ES = (DT == CCL_BF16 || DT == CCL_F16) ? 2 : 4;
    for (long long i = lo + tid; i < hi; i += T) {
        if (ES == 4) {
            unsigned x = __ldcg(reinterpret_cast<const unsigned int*>(a) + i);
            x = add2<DT>(x, __ldcg(reinterpret_cast<const unsigned int*>(b) + i));
            x = add2<DT>(x, __ldcg(reinterpret_cast<const unsigned int*>(c) + i));
            if (o1) __stcg(reinterpret_cast<unsigned int*>(o1) + i, x);
            if (o2) __stcg(reinterpret_cast<unsigned int*>(o2) + i, x);
        } else {
            unsigned x = __ldcg(reinterpret_cast<const unsigned short*>(a) + i);
            x = add2<DT>(x, __ldcg(reinterpret_cast<const unsigned short*>(b) + i)) & 0xffffu;
            x = add2<DT>(x, __ldcg(reinterpret_cast<const unsigned short*>(c) + i)) & 0xffffu;
            if (o1) __stcg(reinterpret_cast<unsigned short*>(o1) + i, (unsigned short)x);
            if (o2) __stcg(reinterpret_cast<unsigned short*>(o2) + i, (unsigned short)x);
        }
    }
}

// o1 (and o2) <- (a + b) + c over n elements, shared by threads [0, T)
template <int DT, int U>
__device__ CCL_MOVE_ATTR void move3(const char* a, bool as, const char* b, bool bs, const char* c, bool cs, char* o1,
                                    bool o1s, char* o2, long long n, int tid, int T)
{
    constexpr int ES = (DT == CCL_BF16 || DT == CCL_F16) ? 2 : 4;
    constexpr int VE = 16 / ES;
    constexpr int U3 = U >= 8 ? 6 : 3;
    const unsigned long long al = (unsigned long long)a | (unsigned long long)b | (unsigned long long)c |
                                  (unsigned long long)o1 | (unsigned long long)o2;
    long long nv = 0;
    if ((al & 15) == 0) {
        nv = n / VE;
        move_vec3<DT, U3>(reinterpret_cast<const uint4*>(a), as, reinterpret_cast<const uint4*>(b), bs,
                          reinterpret_cast<const uint4*>(c), cs, reinterpret_cast<uint4*>(o1), o1s,
                          reinterpret_cast<uint4*>(o2), nv, tid, T);
    }
    if (nv * VE < n) move_elem3<DT>(a, b, c, o1, o2, nv * VE, n, tid, T);
}

// the dtype dispatch of move3 (inlined into the sequential engine's step;
// the pipelined engine's data warps call it out of line, move_part3_call,
// which keeps their two-operand path's registers as they were)
template <int U>
__device__ __forceinline__ void move_part3(int dtype, const char* a, bool as, const char* b, bool bs, const char* c,
                                           bool cs, char* o1, bool o1s, char* o2, long long n, int tid, int T)
{
    switch (dtype) {
    case CCL_F32: move3<CCL_F32, U>(a, as, b, bs, c, cs, o1, o1s, o2, n, tid, T); break;
    case CCL_BF16: move3<CCL_BF16, U>(a, as, b, bs, c, cs, o1, o1s, o2, n, tid, T); break;
    case CCL_F16: move3<CCL_F16, U>(a, as, b, bs, c, cs, o1, o1s, o2, n, tid, T); break;
    default: move3<CCL_I32, U>(a, as, b, bs, c, cs, o1, o1s, o2, n, tid, T); break;
    }
}

template <int U>
__device__ __noinline__ void move_part3_call(int dtype, const char* a, bool as, const char* b, bool bs, const char* c,
                                             bool cs, char* o1, bool o1s, char* o2, long long n, int tid, int T)
{
    move_part3<U>(dtype, a, as, b, bs, c, cs, o1, o1s, o2, n, tid, T);
}

// A copy to three destinations (a folded chain of three direct copies):
// 16-byte vectors when every address allows, else elements of es bytes.
// Inlined into the sequential engine's step; the pipelined engine's data
// warps call it out of line (copy3_call), which keeps their registers.
__device__ __forceinline__ void copy3_part(const char* a, char* o1, char* o2, char* o3, long long n, int es, int tid,
                                           int T)
{
    const unsigned long long al = (unsigned long long)a | (unsigned long long)o1 | (unsigned long long)o2 |
                                  (unsigned long long)o3;
    const long long ve = 16 / es;
    long long nv = 0;
    if ((al & 15) == 0) {
        nv = n / ve;
        const uint4* va = reinterpret_cast<const uint4*>(a);
        uint4* v1 = reinterpret_cast<uint4*>(o1);
        uint4* v2 = reinterpret_cast<uint4*>(o2);
        uint4* v3 = reinterpret_cast<uint4*>(o3);
        long long i = tid;
        for (; i + 3 * (long long)T < nv; i += 4 * (long long)T) {
            uint4 r[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) r[u] = __ldcg(va + i + u * T);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                __stcg(v1 + i + u * T, r[u]);
                __stcg(v2 + i + u * T, r[u]);
                __stcg(v3 + i + u * T, r[u]);
            }
        }
        for (; i < nv; i += T) {
            const uint4 r = __ldcg(va + i);
            __stcg(v1 + i, r);
            __stcg(v2 + i, r);
            __stcg(v3 + i, r);
        }
    }
    for (long long i = nv * ve + tid; i < n; i += T) {
        if (es == 4) {
            const unsigned x = __ldcg(reinterpret_cast<const unsigned*>(a) + i);
            __stcg(reinterpret_cast<unsigned*>(o1) + i, x);
            __stcg(reinterpret_cast<unsigned*>(o2) + i, x);
            __stcg(reinterpret_cast<unsigned*>(o3) + i, x);
        } else {
            const unsigned short x = __ldcg(reinterpret_cast<const unsigned short*>(a) + i);
            __stcg(reinterpret_cast<unsigned short*>(o1) + i, x);
            __stcg(reinterpret_cast<unsigned short*>(o2) + i, x);
            __stcg(reinterpret_cast<unsigned short*>(o3) + i, x);
        }
    }
}

static __device__ __noinline__ void copy3_call(const char* a, char* o1, char* o2, char* o3, long long n, int es, int tid,
                                        int T)
{
    copy3_part(a, o1, o2, o3, n, es, tid, T);
}

// kinds that reduce, and those that take a third operand (held in the
// source range)
__device__ __forceinline__ bool kind_reduces(int k)
{
    return k == CCL_I_REDUCE || k == CCL_I_RRC || k == CCL_I_RRS || k == CCL_I_RRCS || k == CCL_I_RRC2 ||
           k == CCL_I_RRS3 || k == CCL_I_RRC3 || k == CCL_I_RRCS3 || k == CCL_I_RSEND || k == CCL_I_RCSEND ||
           k == CCL_I_RRC3D || k == CCL_I_REDUCE2;
}
__device__ __forceinline__ bool kind_three(int k)
{
    return k == CCL_I_RRS3 || k == CCL_I_RRC3 || k == CCL_I_RRCS3 || k == CCL_I_RRC3D;
}

// the whole CTA moves the data
template <int DT>
__device__ __forceinline__ void move_dt(bool red, const char* a, bool as, const char* b, bool bs, char* o1,
                                        bool o1s, char* o2, long long n)
{
    move_part<DT, 4>(red, a, as, b, bs, o1, o1s, o2, n, threadIdx.x, blockDim.x);
}

// vectors in flight per operand per thread for a kernel built for at most
// MAXT threads
template <int MAXT>
struct InFlight {
    static constexpr int U = MAXT <= 512 ? 8 : 4;
};

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

// ----------------------------------------------------------------------
// Warp-specialised executor.  Four roles per CTA:
//
//  * issuer (warp 0, lane 0) walks the threadblock program.  Step records
//    (144 bytes each) arrive by cp.async in batches of kLook, one batch
//    ahead.  It waits (bounded) for the first slot of up to kLook coming
//    steps -- incoming slot full, outgoing slot free -- and for their first
//    kDepPoll dependency counters, polling all those words with relaxed
//    loads in one round trip, then one acquire fence; later slots of a step
//    are polled kBatch at a time, further counters one step at a time.  A step that follows an earlier step of its own threadblock
//    waits only for that step's last tile.  Slots are handed out as tiles
//    of at most `tile` bytes through a ring of kQ shared-memory descriptors
//    guarded by mbarriers ("ready").  Slot indices are computed in 32 bits
//    from residues the plan precomputes (no 64-bit division on one thread).
//  * TMA thread (warp 2, lane 0) moves every 16-byte-aligned *copy* tile
//    with bulk copies: global -> shared stage (mbarrier complete_tx), then
//    shared -> global to the destination and/or the outgoing slot (bulk
//    groups).  Up to `ns` tiles are in flight; a stage is reused once its
//    stores have read it, and a tile counts as done once its stores are
//    complete.
//  * data warps (warps 3..) move the other tiles (every reduce, and copies
//    that are not 16-byte aligned) with 16-byte / element loads and stores;
//    in the LL instantiation they also poll incoming LL lines and write
//    outgoing lines with the slot's flag.
//  * releaser (warp 1, lane 0) takes finished tiles in order, issues one
//    release fence per batch and posts the flags and counters carried by a
//    slot's last tile with relaxed stores, then frees the descriptor.
//
// Both the TMA thread and the data warps acknowledge every descriptor (the
// one that moves a tile once it is moved, the other as soon as it has seen
// that the tile is not its own), and a descriptor is reused only after both
// acknowledgements, so no role ever misses a descriptor.
// ----------------------------------------------------------------------
constexpr int kQ = 16;     // tile descriptors in flight
constexpr int kNSMax = 8;  // shared-memory stages
constexpr int kRetireDepth = 7;   // store groups left in flight when retiring
constexpr int kCQ = 16;           // stored tiles awaiting completion (> kRetireDepth)
// last descriptor of each of the latest kHist steps; every step hands out at
// least one descriptor and descriptors are freed in order, so a step further
// back than kQ + 1 steps is finished whenever the issuer runs
constexpr int kHist = 32;
static_assert(kHist > kQ, "history must reach past the descriptor ring");

struct SlotOp {
    const char* a;      // data in: incoming slot or source buffer
    const char* b;      // local operand of a reduce
    const char* c;      // third operand (a folded reduction chain), or null
    char* o1;           // destination buffer, or the outgoing slot
    char* o2;           // outgoing slot when a destination is also written
    char* o3;           // third destination (a folded chain of three copies), or null
    long long n;        // elements
    int red, dtype;
    int as, bs, cs, o1s;   // streaming cache hints (register path)
    int bulk;           // moved by the TMA thread
    int cmd;            // 0 move, 1 end, 2 abort
    int a_ll, o1_ll, o2_ll;   // operand is an LL slot
    unsigned fin, fout;       // flag of the incoming / outgoing LL slot
};

struct Release {
    unsigned long long* consumed;  // flag to post, or null
    unsigned long long* full;
    unsigned long long* counter;
    unsigned long long consumed_v, full_v, counter_v;
    unsigned long long t_start, waited, t_pub;
    int si;
    int last;                      // last tile of its step
};

// steps whose first-slot flags and first kDepPoll dependency counters the
// issuer polls in one round trip
constexpr int kLook = 4;
constexpr int kDepPoll = 2;

struct CtlShared {
    DRec rec[2 * kLook];                // two batches of step records (prefetched one batch ahead)
    SlotOp op[kQ];
    Release rel[kQ];
    unsigned long long ready[kQ];
    unsigned long long done_g[kQ];      // data warps are through with the descriptor
    unsigned long long done_b[kQ];      // the TMA thread is through with the descriptor
    unsigned long long freed[kQ];
    unsigned long long full[kNSMax];    // stage loaded
    int last_head[kHist];               // issuer only: last descriptor of step si % kHist
    const unsigned long long* poll_ptr[kLook * (2 + kDepPoll)];   // issuer only: polled words
    unsigned long long poll_want[kLook * (2 + kDepPoll)];         // and their targets
    DLink links[kSeqLinks];             // the program's first links (KParams.prog_links)
};

// A step's link: the program's copy in shared memory when the record says
// where (link_loc), else the link array
__device__ __forceinline__ const DLink* step_link(const KParams& P, const DLink* tab, int link, int loc)
{
    return link < 0 ? nullptr : loc ? tab + (loc - 1) : P.links + link;
}
// copy the program's first links into shared memory (threads < kSeqLinks)
__device__ __forceinline__ void load_prog_links(const KParams& P, int prog, DLink* tab)
{
    if (threadIdx.x < kSeqLinks) {
        const int id = P.prog_links[prog * kSeqLinks + threadIdx.x];
        if (id >= 0) tab[threadIdx.x] = P.links[id];
    }
}

__device__ __forceinline__ void record_timeout(const KParams& P, int si, int reason)
{
    if (atomicCAS(P.status, 0, (int)CCL_ERR_TIMEOUT) == 0) {
        P.status[1] = blockIdx.x;
        P.status[2] = si;
        P.status[3] = reason;
    }
}

// bounded wait on an mbarrier phase inside the CTA: try_wait suspends the
// thread in hardware until the phase completes or a short time passes
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, unsigned par, unsigned long long limit_ns)
{
    unsigned long long t0 = 0;
    while (!mbar_try_wait(bar, par)) {
        const unsigned long long now = gtimer();
        if (!t0) t0 = now;
        else if (now - t0 > limit_ns) return false;
    }
    return true;
}

// Bounded wait until every dependency counter of a step reaches its value:
// up to kDepBatch counters polled with relaxed loads issued together per
// round trip, one acquire fence at the end.
constexpr int kDepBatch = 8;
static __device__ bool wait_deps(const KParams& P, const DDep* deps, int n, int si, unsigned long long& waited,
                                 bool acq1 = false)
{
    const unsigned long long base = (unsigned long long)(P.exec * P.m);
    unsigned long long t0 = 0;
    if (n == 1 && acq1) {
        // one counter (the sequential engine): acquire loads, no separate
        // fence
        const unsigned long long* c = P.counters + deps[0].counter;
        const unsigned long long v = base + deps[0].value;
        unsigned spins = 0;
        while (ld_acquire(c) < v) {
            if (!t0) t0 = gtimer();
            ++spins;
            if ((spins & 15) == 0) {
                if (*(volatile int*)P.status != 0) return false;
                if (gtimer() - t0 > P.timeout_ns) {
                    record_timeout(P, si, WAIT_DEP);
                    return false;
                }
            }
            if (spins > 64) __nanosleep(32);
        }
        if (t0) waited += gtimer() - t0;
        return true;
    }
    for (int k0 = 0; k0 < n; k0 += kDepBatch) {
        const int nb = n - k0 < kDepBatch ? n - k0 : kDepBatch;
        const unsigned long long* c[kDepBatch];
        unsigned long long v[kDepBatch];
#pragma unroll
        for (int i = 0; i < kDepBatch; ++i) {
            const DDep d = deps[k0 + (i < nb ? i : 0)];
            c[i] = P.counters + d.counter;
            v[i] = base + d.value;
        }
        unsigned spins = 0;
        while (true) {
            bool ok = true;
#pragma unroll
            for (int i = 0; i < kDepBatch; ++i)
                if (i < nb && ld_relaxed(c[i]) < v[i]) ok = false;
            if (ok) break;
            if (!t0) t0 = gtimer();
            ++spins;
            if ((spins & 15) == 0) {
                if (*(volatile int*)P.status != 0) return false;
                if (gtimer() - t0 > P.timeout_ns) {
                    record_timeout(P, si, WAIT_DEP);
                    return false;
                }
            }
            if (spins > 64) __nanosleep(32);
        }
    }
    fence_acq_rel_gpu();
    if (t0) waited += gtimer() - t0;
    return true;
}

// Batched form for consecutive slots k .. k+bmax-1 of one step: the flags of
// all of them are polled with relaxed loads in one round trip; returns how
// many leading slots are ready (>= 1), after one acquire fence, or 0 when the
// wait for the first one fails.  out_rel0: the outgoing sequence of slot k
// counted from the start of this execution.
constexpr int kBatch = 4;
static __device__ int wait_slots(const KParams& P, const DLink* Lin, const DLink* Lout, unsigned long long sin0,
                          unsigned long long sout0, long long out_rel0, unsigned in_idx0, unsigned out_idx0, int bmax,
                          int si, unsigned long long& waited, bool acq1 = false)
{
    const unsigned S = (unsigned)P.S;
    // nothing to poll (an LL or absent incoming link, outgoing slots first
    // used in this execution -- last read in an earlier one, a finished
    // kernel): every slot is ready, with no fence
    const bool poll_in = Lin && !P.ll;
    const bool poll_out = Lout && out_rel0 + bmax - 1 >= (long long)P.S;
    if (!poll_in && !poll_out) return bmax;
    unsigned long long t0 = 0;
    unsigned spins = 0;
    if (acq1 && bmax == 1 && poll_in != poll_out) {
        // one word (the sequential engine): acquire loads, no separate fence
        const unsigned long long* w = poll_in ? P.flags + Lin->flag_base + in_idx0
                                              : P.flags + Lout->flag_base + S + out_idx0;
        const unsigned long long v = poll_in ? sin0 + 1 : sout0 + 1 - P.S;
        while (ld_acquire(w) < v) {
            if (!t0) t0 = gtimer();
            ++spins;
            if ((spins & 15) == 0) {
                if (*(volatile int*)P.status != 0) return 0;
                if (gtimer() - t0 > P.timeout_ns) {
                    record_timeout(P, si, poll_in ? WAIT_FULL : WAIT_FREE);
                    return 0;
                }
            }
            if (spins > 64) __nanosleep(32);
        }
        if (t0) waited += gtimer() - t0;
        return 1;
    }
    while (true) {
        unsigned long long x[kBatch], y[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            x[i] = ~0ull;
            y[i] = ~0ull;
            if (i < bmax) {
                unsigned ii = in_idx0 + i, io = out_idx0 + i;   // slot indices: i < kBatch, S >= 2
                while (ii >= S) ii -= S;
                while (io >= S) io -= S;
                if (poll_in) x[i] = ld_relaxed(P.flags + Lin->flag_base + ii);
                if (Lout && out_rel0 + i >= (long long)P.S) y[i] = ld_relaxed(P.flags + Lout->flag_base + S + io);
            }
        }
        int b = 0;
        while (b < bmax && x[b] >= sin0 + b + 1 && y[b] >= sout0 + b + 1 - P.S) ++b;
        if (b > 0) {
            fence_acq_rel_gpu();
            if (t0) waited += gtimer() - t0;
            return b;
        }
        if (!t0) t0 = gtimer();
        ++spins;
        if ((spins & 15) == 0) {
            if (*(volatile int*)P.status != 0) return 0;
            if (gtimer() - t0 > P.timeout_ns) {
                record_timeout(P, si, x[0] < sin0 + 1 ? WAIT_FULL : WAIT_FREE);
                return 0;
            }
        }
        if (spins > 64) __nanosleep(32);
    }
}

__device__ __forceinline__ void prefetch_rec(DRec* dst, const DRec* src)
{
    const unsigned d = smem_addr(dst);
#pragma unroll
    for (int k = 0; k < (int)(sizeof(DRec) / 16); ++k)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d + 16 * k), "l"((const char*)src + 16 * k)
                     : "memory");
}

// flag word and value that say the first FIFO slot of a step may be read
// (incoming slot full) or written (outgoing slot consumed S sequences ago)
struct SlotCond {
    const unsigned long long* in;
    const unsigned long long* out;
    unsigned long long vin, vout;
};

// slot index (sequence % S) of a step's first slot on link L, in 32 bits:
// (exec * total + seq) % S from exec % S, total % S and seq % S
__device__ __forceinline__ unsigned slot_index(unsigned exec_mod, const DLink& L, int seq_mod, unsigned S)
{
    return (exec_mod * (unsigned)L.total_mod + (unsigned)seq_mod) % S;
}

// Lin / Lout: the step's links (null when absent)
__device__ __forceinline__ SlotCond first_slot_cond(const KParams& P, const DRec& st, unsigned exec_mod,
                                                    const DLink* Lin, const DLink* Lout)
{
    SlotCond c{nullptr, nullptr, 0, 0};
    const unsigned S = (unsigned)P.S;
    if (Lin && !P.ll) {   // LL: the data path polls the lines
        const DLink& L = *Lin;
        const unsigned long long s = (unsigned long long)(P.exec * L.total) + st.seq_in;
        c.in = P.flags + L.flag_base + slot_index(exec_mod, L, st.seq_in_mod, S);
        c.vin = s + 1;
    }
    // the slot's previous use: in an earlier execution (a finished kernel:
    // nothing to wait for) unless this execution has used S slots already
    if (Lout && st.seq_out >= (long long)P.S) {
        const DLink& L = *Lout;
        const unsigned long long s = (unsigned long long)(P.exec * L.total) + st.seq_out;
        c.out = P.flags + L.flag_base + S + slot_index(exec_mod, L, st.seq_out_mod, S);
        c.vout = s + 1 - P.S;
    }
    return c;
}

__device__ __forceinline__ SlotCond first_slot_cond(const KParams& P, const DRec& st, unsigned exec_mod,
                                                    const DLink* tab)
{
    return first_slot_cond(P, st, exec_mod, step_link(P, tab, st.link_in, st.link_loc & 0xff),
                           step_link(P, tab, st.link_out, (st.link_loc >> 8) & 0xff));
}

// Poll the conditions of steps [s0, s1) (records in the ring) -- the first
// FIFO slot's flags and the first kDepPoll dependency counters of each --
// with relaxed loads issued together; returns the end of the leading run of
// ready steps (> s0) after one acquire fence, or -1 when the wait for step
// s0 fails.  Counters of a step beyond kDepPoll are left to wait_deps.
static __device__ int poll_steps(const KParams& P, CtlShared* sh, int s0, int s1, unsigned exec_mod,
                          unsigned long long& waited)
{
    constexpr int kC = 2 + kDepPoll;   // conditions per step
    const int n = s1 - s0;
    const unsigned long long base = (unsigned long long)(P.exec * P.m);
    // condition words and targets go to shared memory (the issuer's
    // registers are capped with the rest of the kernel's)
#pragma unroll
    for (int i = 0; i < kLook; ++i) {
        const unsigned long long** ptr = sh->poll_ptr + i * kC;
        unsigned long long* want = sh->poll_want + i * kC;
        if (i >= n) {
            for (int k = 0; k < kC; ++k) ptr[k] = nullptr;
            continue;
        }
        const DRec& st = sh->rec[(s0 + i) % (2 * kLook)];
        const SlotCond c = first_slot_cond(P, st, exec_mod, sh->links);
        ptr[0] = c.in;
        want[0] = c.vin;
        ptr[1] = c.out;
        want[1] = c.vout;
        for (int k = 0; k < kDepPoll; ++k) {
            if (k < st.dep_count) {
                const DDep d = P.deps[st.dep_begin + k];
                ptr[2 + k] = P.counters + d.counter;
                want[2 + k] = base + d.value;
            } else {
                ptr[2 + k] = nullptr;
            }
        }
    }
    unsigned long long t0 = 0;
    unsigned spins = 0;
    while (true) {
        unsigned long long x[kLook * kC];
#pragma unroll
        for (int k = 0; k < kLook * kC; ++k) {
            const unsigned long long* q = sh->poll_ptr[k];
            x[k] = q ? ld_relaxed(q) : ~0ull;
        }
        int r = 0;
        bool ok = true;
#pragma unroll
        for (int i = 0; i < kLook; ++i) {
#pragma unroll
            for (int k = 0; k < kC; ++k)
                if (x[i * kC + k] < sh->poll_want[i * kC + k]) ok = false;
            if (ok && i < n) r = i + 1;
        }
        if (r > 0) {
            fence_acq_rel_gpu();
            if (t0) waited += gtimer() - t0;
            return s0 + r;
        }
        if (!t0) t0 = gtimer();
        ++spins;
        if ((spins & 15) == 0) {
            if (*(volatile int*)P.status != 0) return -1;
            if (gtimer() - t0 > P.timeout_ns) {
                record_timeout(P, s0, x[0] < sh->poll_want[0]   ? WAIT_FULL
                                      : x[1] < sh->poll_want[1] ? WAIT_FREE
                                                                : WAIT_DEP);
                return -1;
            }
        }
        if (spins > 64) __nanosleep(32);
    }
}

__device__ __forceinline__ bool aligned16(const void* p) { return ((unsigned long long)p & 15) == 0; }

// publish a command descriptor (1 end, 2 abort) behind every tile handed out
__device__ __forceinline__ void publish_cmd(CtlShared* sh, int head, int cmd, unsigned long long limit)
{
    const int q = head % kQ;
    if (head >= kQ) mbar_wait(&sh->freed[q], (unsigned)(((head / kQ) - 1) & 1), limit);
    sh->op[q].cmd = cmd;
    mbar_arrive(&sh->ready[q]);
}

// Wait (bounded) until every tile of step `drain` of this threadblock has
// been released: its last descriptor, and, freed in order, all earlier ones.
// Steps further back than kHist are finished whenever the issuer runs.
__device__ __forceinline__ bool wait_drain(const KParams& P, CtlShared* sh, int drain, int si, int head)
{
    if (drain < 0 || si - drain >= kHist) return true;
    const int h = sh->last_head[drain % kHist];
    if (h >= head - kQ && !mbar_wait(&sh->freed[h % kQ], (unsigned)((h / kQ) & 1), 4 * P.timeout_ns)) {
        record_timeout(P, si, WAIT_DONE);
        return false;
    }
    return true;
}

// Hand the slots of step si out to the data path as tile descriptors (the
// common part of the issuer that walks the step records and of the issuers
// generated for single plans).  Its dependency counters and drain are
// already satisfied; ready_slots leading slots were already seen ready, the
// others are polled kBatch at a time.  Lin / Lout: the step's links (null
// when absent).  False after a failed wait (the abort command is then
// published).
__device__ __forceinline__ bool issue_step(const KParams& P, CtlShared* sh, const DRec& st, const DLink* Lin,
                                           const DLink* Lout, int si, int& head, int ready_slots,
                                           unsigned exec_mod, unsigned long long t_start,
                                           unsigned long long& waited)
{
    const unsigned long long limit = 4 * P.timeout_ns;
    const unsigned S = (unsigned)P.S;
    unsigned long long t_pub = 0;
    const int es = (st.dtype == CCL_BF16 || st.dtype == CCL_F16) ? 2 : 4;
    const unsigned long long base_in = Lin ? (unsigned long long)(P.exec * Lin->total) : 0;
    const unsigned long long base_out = Lout ? (unsigned long long)(P.exec * Lout->total) : 0;
    const int esh = es == 2 ? 1 : 2;
    const long long slot_elems = P.slot_bytes >> esh;
    // tiles exist for the bulk path; the register path takes a slot whole
    const long long tile_elems = (P.ns > 0 ? P.tile_bytes : P.slot_bytes) >> esh;
    const bool linked = Lin || Lout;
    // FIFO slots of a linked step; local steps are cut into tiles directly
    long long nslots = linked ? (st.nslots > 0 ? st.nslots : 1) : 1;
    if (!linked && st.nelem > 0)
        nslots = st.nelem + tile_elems - 1 < 0xffffffffll
                     ? (unsigned)(st.nelem + tile_elems - 1) / (unsigned)tile_elems
                     : (st.nelem + tile_elems - 1) / tile_elems;
    unsigned in_idx = Lin ? slot_index(exec_mod, *Lin, st.seq_in_mod, S) : 0;
    unsigned out_idx = Lout ? slot_index(exec_mod, *Lout, st.seq_out_mod, S) : 0;
    const long long span = linked ? slot_elems : tile_elems;
    const int red = kind_reduces(st.kind);
    const bool three = kind_three(st.kind);
    const char* srcb = st.src_buf >= 0 ? P.bufs[st.src_buf][st.src_rank] + st.src_off * es : nullptr;
    const char* locb = st.loc_buf >= 0 ? P.bufs[st.loc_buf][st.loc_rank] + st.loc_off * es : nullptr;
    char* dstb = st.dst_buf >= 0 ? P.bufs[st.dst_buf][st.dst_rank] + st.dst_off * es : nullptr;
    const bool post = !(st.flags & STEP_NOPOST);
    for (long long k = 0; k < nslots; ++k) {
        const unsigned long long sin = base_in + st.seq_in + k;
        const unsigned long long sout = base_out + st.seq_out + k;
        if (linked && ready_slots == 0) {
            const int bmax = (int)((nslots - k) < kBatch ? (nslots - k) : kBatch);
            ready_slots = wait_slots(P, Lin, Lout, sin, sout, st.seq_out + k, in_idx, out_idx, bmax, si, waited);
            if (ready_slots == 0) {
                publish_cmd(sh, head, 2, limit);
                return false;
            }
        }
        if (linked) --ready_slots;
        const long long e0 = k * span;
        long long n = st.nelem - e0;
        if (n > span) n = span;
        if (n < 0) n = 0;
        const char* slot_in = Lin ? P.fifo + Lin->slot_base + (long long)in_idx * P.slot_stride : nullptr;
        char* slot_out = Lout ? P.fifo + Lout->slot_base + (long long)out_idx * P.slot_stride : nullptr;
        const long long lls = P.ll ? 2 : 1;   // slot bytes per data byte
        // n <= slot_elems: 32-bit division
        const long long ntiles = n > 0 ? (long long)((unsigned)(n + tile_elems - 1) / (unsigned)tile_elems) : 1;
        for (long long u = 0; u < ntiles; ++u) {
            const int q = head % kQ;
            if (head >= kQ && !mbar_wait(&sh->freed[q], (unsigned)(((head / kQ) - 1) & 1), limit)) {
                record_timeout(P, si, WAIT_DONE);
                publish_cmd(sh, head, 2, limit);
                return false;
            }
            const long long t0 = u * tile_elems;
            long long tn = n - t0;
            if (tn > tile_elems) tn = tile_elems;
            if (tn < 0) tn = 0;
            const long long off = (e0 + t0) * es;   // byte offset in the step's buffers
            const long long soff = t0 * es;         // byte offset in the slot
            SlotOp& op = sh->op[q];
            op.a_ll = op.o1_ll = op.o2_ll = 0;
            if (Lin && st.kind != CCL_I_REDUCE) {
                op.a = slot_in + lls * soff;
                op.as = 0;
                op.a_ll = P.ll;
            } else {
                op.a = srcb + off;
                op.as = (st.flags & STEP_SRC_STREAM) && P.stream_in;
            }
            // a two-destination copy keeps its second destination in the
            // local-operand range
            // (a folded recv-reduce-copy-send: in its source range)
            const bool copy2 = st.kind == CCL_I_COPY2 || st.kind == CCL_I_COPY3, rrc2 = st.kind == CCL_I_RRC2;
            op.b = locb && !copy2 ? locb + off : nullptr;
            op.o3 = st.kind == CCL_I_COPY3 ? P.bufs[st.x_buf][st.x_rank] + st.x_off * es + off : nullptr;
            op.bs = (st.flags & STEP_LOC_STREAM) && P.stream_in;
            // a folded reduction chain's third operand: its source range
            op.c = three && srcb ? srcb + off : nullptr;
            op.cs = (st.flags & STEP_SRC_STREAM) && P.stream_in;
            if (dstb) {
                op.o1 = dstb + off;
                op.o1s = st.dst_buf == CCL_BUF_OUT;
                // (a second destination -- a folded receive -- is written
                // instead of a slot)
                op.o2 = copy2  ? const_cast<char*>(locb) + off
                        : rrc2 ? const_cast<char*>(srcb) + off
                        : st.x_buf >= 0 ? P.bufs[st.x_buf][st.x_rank] + st.x_off * es + off
                        : slot_out ? slot_out + lls * soff
                                   : nullptr;
                op.o2_ll = slot_out && P.ll;
            } else {
                op.o1 = slot_out + lls * soff;
                op.o1s = 0;
                op.o2 = nullptr;
                op.o1_ll = P.ll;
            }
            op.fin = (unsigned)(sin + 1);
            op.fout = (unsigned)(sout + 1);
            op.n = tn;
            op.red = red;
            op.dtype = st.dtype;
            op.bulk = P.ns > 0 && !red && !op.o3 && tn > 0 && ((tn * es) & 15) == 0 && aligned16(op.a) &&
                      aligned16(op.o1) && (!op.o2 || aligned16(op.o2)) && !op.a_ll && !op.o1_ll && !op.o2_ll;
            op.cmd = 0;
            Release& r = sh->rel[q];
            const bool last_tile = u == ntiles - 1;
            // a consumed flag matters only to a producer that reuses the slot
            // within this execution (S sequences later)
            r.consumed = (Lin && post && last_tile && st.seq_in + k + S < Lin->total)
                             ? P.flags + Lin->flag_base + S + in_idx
                             : nullptr;
            r.consumed_v = sin + 1;
            // LL slots carry their flags in the lines
            r.full = (Lout && post && last_tile && !P.ll) ? P.flags + Lout->flag_base + out_idx : nullptr;
            r.full_v = sout + 1;
            r.last = last_tile && k == nslots - 1;
            r.counter = (st.signal >= 0 && post) ? P.counters + st.signal : nullptr;
            r.counter_v = (unsigned long long)(P.exec * P.m + st.mb + 1);
            r.si = si;
            if (P.timeline && !t_pub) t_pub = gtimer();
            r.t_start = t_start;
            r.waited = waited;
            r.t_pub = t_pub;
            mbar_arrive(&sh->ready[q]);
            ++head;
        }
        if (++in_idx == S) in_idx = 0;
        if (++out_idx == S) out_idx = 0;
    }
    sh->last_head[si % kHist] = head - 1;
    return true;
}

// The issuer of the library's kernel: walks the threadblock's step records.
static __device__ void issuer(const KParams& P, CtlShared* sh, int b0, int b1)
{
    int head = 0;
    const unsigned long long limit = 4 * P.timeout_ns;
    // records arrive in batches of kLook, one batch ahead: [rec_ready,
    // rec_end) is in flight, everything below rec_ready is in shared memory
    int rec_ready = b0, rec_end = b0;
    auto request = [&](int from) {
        rec_end = from + kLook < b1 ? from + kLook : b1;
        for (int j = from; j < rec_end; ++j) prefetch_rec(&sh->rec[j % (2 * kLook)], P.recs + j);
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    if (b0 < b1) request(b0);
    int cleared = b0;   // steps below: first-slot flags seen ready (and fenced)
    // slot indices in 32-bit arithmetic: no 64-bit division on the way to a
    // step (the issuer is one thread; a 64-bit modulo is a long routine)
    const unsigned exec_mod = (unsigned)(P.exec % P.S);
    for (int si = b0; si < b1; ++si) {
        if (si >= rec_ready) {
            asm volatile("cp.async.wait_all;" ::: "memory");
            rec_ready = rec_end;
            if (rec_end < b1) request(rec_end);
        }
        const DRec& st = sh->rec[si % (2 * kLook)];
        const unsigned long long t_start = gtimer();
        unsigned long long waited = 0;
        if (si >= cleared) {
            // one round trip for the first-slot flags and dependency
            // counters of the next steps whose records are here
            const int s1 = rec_ready < si + kLook ? rec_ready : si + kLook;
            cleared = poll_steps(P, sh, si, s1, exec_mod, waited);
            if (cleared < 0) {
                publish_cmd(sh, head, 2, limit);
                return;
            }
        }
        // reads or writes what an earlier step of this threadblock touched
        if (!wait_drain(P, sh, st.drain, si, head)) {
            publish_cmd(sh, head, 2, limit);
            return;
        }
        if (st.dep_count > kDepPoll &&
            !wait_deps(P, P.deps + st.dep_begin + kDepPoll, st.dep_count - kDepPoll, si, waited)) {
            publish_cmd(sh, head, 2, limit);
            return;
        }
        const DLink* Lin = step_link(P, sh->links, st.link_in, st.link_loc & 0xff);
        const DLink* Lout = step_link(P, sh->links, st.link_out, (st.link_loc >> 8) & 0xff);
        if (!issue_step(P, sh, st, Lin, Lout, si, head, si < cleared ? 1 : 0, exec_mod, t_start, waited)) return;
    }
    publish_cmd(sh, head, 1, limit);
}

static __device__ void releaser(const KParams& P, CtlShared* sh)
{
    const unsigned long long limit = 4 * P.timeout_ns;
    for (int j = 0;;) {
        int q = j % kQ;
        unsigned par = (unsigned)((j / kQ) & 1);
        if (!mbar_wait(&sh->ready[q], par, limit)) {
            record_timeout(P, -1, WAIT_DONE);
            return;
        }
        if (sh->op[q].cmd != 0) return;
        if (!mbar_wait(&sh->done_g[q], par, limit) || !mbar_wait(&sh->done_b[q], par, limit)) {
            record_timeout(P, -1, WAIT_DONE);
            return;
        }
        // batch every further tile that is already finished
        int n = 1;
        while (n < kQ) {
            const int q2 = (j + n) % kQ;
            const unsigned p2 = (unsigned)(((j + n) / kQ) & 1);
            if (!mbar_test(&sh->ready[q2], p2) || sh->op[q2].cmd != 0) break;
            if (!mbar_test(&sh->done_g[q2], p2) || !mbar_test(&sh->done_b[q2], p2)) break;
            ++n;
        }
        const unsigned long long t_done = P.timeline ? gtimer() : 0;
        fence_acq_rel_gpu();
        for (int i = 0; i < n; ++i) {
            const Release& r = sh->rel[(j + i) % kQ];
            if (r.consumed) st_relaxed(r.consumed, r.consumed_v);
            if (r.full) st_relaxed(r.full, r.full_v);
            if (r.last) {
                if (r.counter) st_relaxed(r.counter, r.counter_v);
                if (P.timeline) {
                    unsigned long long* tl = P.timeline + 5ll * r.si;
                    tl[0] = r.t_start;
                    tl[1] = r.waited;
                    tl[2] = r.t_pub;
                    tl[3] = t_done;
                    tl[4] = gtimer();
                }
            }
        }
        for (int i = 0; i < n; ++i) mbar_arrive(&sh->freed[(j + i) % kQ]);
        j += n;
    }
}

// TMA thread: bulk copies of aligned copy tiles through the shared-memory
// stages; every other descriptor is acknowledged at once
static __device__ void tma_thread(const KParams& P, CtlShared* sh, unsigned char* stages)
{
    const int NS = P.ns;
    if (NS == 0) {
        // bulk path off: acknowledge every descriptor as it comes
        for (int j = 0;; ++j) {
            const int q = j % kQ;
            if (!mbar_wait(&sh->ready[q], (unsigned)((j / kQ) & 1), 4 * P.timeout_ns)) {
                record_timeout(P, -1, WAIT_DONE);
                return;
            }
            if (sh->op[q].cmd != 0) return;
            mbar_arrive(&sh->done_b[q]);
        }
    }
    const long long TB = P.tile_bytes;
    const unsigned long long limit = 4 * P.timeout_ns;
    struct Fly { int q, s, tnum; char* o1; char* o2; unsigned bytes; };
    Fly fly[kNSMax];
    int stage_grp[kNSMax];
    for (int i = 0; i < kNSMax; ++i) stage_grp[i] = -1;
    int cq[kCQ] = {};         // tiles stored, waiting for their stores to complete
    int cg[kCQ] = {};
    int c_head = 0, c_tail = 0;
    int j = 0, t = 0, g = 0, f_head = 0, f_tail = 0;
    bool ended = false;
    auto retire = [&](int depth) {
        // all but the newest `depth` store groups are complete
        bulk_wait(depth);
        bool any = false;
        while (c_tail < c_head && cg[c_tail % kCQ] < g - depth) {
            if (!any) { fence_proxy_async_global(); any = true; }
            mbar_arrive(&sh->done_b[cq[c_tail % kCQ]]);
            ++c_tail;
        }
    };
    // leave only when no bulk copy still reads or writes this CTA's shared
    // memory: wait (bounded) for every issued load, then for every store
    auto leave = [&]() {
        for (int i = f_tail; i < f_head; ++i) {
            const Fly& e = fly[i % kNSMax];
            mbar_wait(&sh->full[e.s], (unsigned)((e.tnum / NS) & 1), P.timeout_ns);
        }
        bulk_wait(0);
    };
    auto wait_ready = [&](unsigned long long* bar, unsigned par) {
        unsigned spins = 0;
        unsigned long long t0 = 0;
        while (!mbar_test(bar, par)) {
            if ((++spins & 127) == 0) {
                if (*(volatile int*)P.status != 0) return false;
                unsigned long long now = gtimer();
                if (!t0) t0 = now;
                else if (now - t0 > limit) return false;
            }
            if (spins > 32) __nanosleep(20);
        }
        return true;
    };
    unsigned iter = 0;
    while (true) {
        if ((++iter & 63) == 0 && *(volatile int*)P.status != 0) {
            leave();
            return;
        }
        // 1. start loads of newly handed-out tiles while a stage is free
        while (!ended && f_head - f_tail < NS) {
            const int q = j % kQ;
            if (!mbar_test(&sh->ready[q], (unsigned)((j / kQ) & 1))) break;
            const SlotOp& op = sh->op[q];
            if (op.cmd != 0) { ended = true; break; }
            if (!op.bulk) {
                // not ours: acknowledge right away
                mbar_arrive(&sh->done_b[q]);
                ++j;
                continue;
            }
            const int s = t % NS;
            if (stage_grp[s] >= 0) bulk_wait_read(g - stage_grp[s] - 1);
            const int es = (op.dtype == CCL_BF16 || op.dtype == CCL_F16) ? 2 : 4;
            const unsigned bytes = (unsigned)(op.n * es);
            unsigned char* A = stages + s * TB;
            if (!op.as) fence_proxy_async_global();   // reads data another CTA published
            mbar_arrive_expect_tx(&sh->full[s], bytes);
            bulk_load(A, op.a, bytes, &sh->full[s]);
            fly[f_head % kNSMax] = Fly{q, s, t, op.o1, op.o2, bytes};
            ++f_head;
            ++t;
            ++j;
        }
        if (f_tail < f_head) {
            // 2. store the oldest tile once its load has landed
            const Fly e = fly[f_tail % kNSMax];
            if (!wait_ready(&sh->full[e.s], (unsigned)((e.tnum / NS) & 1))) {
                record_timeout(P, -1, WAIT_DONE);
                leave();
                return;
            }
            const unsigned char* A = stages + e.s * TB;
            bulk_store(e.o1, A, e.bytes);
            if (e.o2) bulk_store(e.o2, A, e.bytes);
            bulk_commit();
            stage_grp[e.s] = g;
            cq[c_head % kCQ] = e.q;
            cg[c_head % kCQ] = g;
            ++c_head;
            ++g;
            ++f_tail;
            if (c_head - c_tail > kRetireDepth) retire(kRetireDepth);
        } else {
            // 3. nothing in flight: finish every store, then wait for work
            retire(0);
            if (ended) return;
            if (!wait_ready(&sh->ready[j % kQ], (unsigned)((j / kQ) & 1))) {
                record_timeout(P, -1, WAIT_DONE);
                leave();
                return;
            }
        }
    }
}

// Copy or reduce a tile of which some operand is an LL slot (16-byte
// multiples, every pointer 16-byte aligned: the plan guarantees it).  An LL
// source is polled line by line until every line carries the slot's flag;
// LL destinations get the data with the outgoing slot's flag.  Returns false
// when a wait gives up (time limit, or another role recorded a failure).
template <bool RED, int DT>
__device__ __forceinline__ bool move_ll(const SlotOp& op, int tid, int T, unsigned long long timeout_ns,
                                        const int* status)
{
    constexpr int ES = (DT == CCL_BF16 || DT == CCL_F16) ? 2 : 4;
    const long long nv = op.n * ES / 16;
    const char* a = op.a;
    const uint4* a16 = reinterpret_cast<const uint4*>(a);
    const uint4* b16 = reinterpret_cast<const uint4*>(op.b);
    const bool a_ll = op.a_ll, o1_ll = op.o1_ll, o2_ll = op.o2_ll, as = op.as, bs = op.bs, o1s = op.o1s;
    char* o1 = op.o1;
    char* o2 = op.o2;
    const unsigned fin = op.fin, fout = op.fout;
    // two vectors in flight per thread: i and i + T
    for (long long i = tid; i < nv; i += 2ll * T) {
        const long long j1 = i + T < nv ? i + T : nv - 1;   // past the end: re-read, never used
        uint4 va0, va1, vb0, vb1;
        if (a_ll) {
            unsigned long long p0, p1, p2, p3, q0, q1, q2, q3;
            ll_load2(a + 32 * i, p0, p1);
            ll_load2(a + 32 * i + 16, p2, p3);
            ll_load2(a + 32 * j1, q0, q1);
            ll_load2(a + 32 * j1 + 16, q2, q3);
            if (RED) {
                vb0 = vload(b16 + i, bs);
                vb1 = vload(b16 + j1, bs);
            }
            unsigned long long t0 = 0;
            unsigned spins = 0;
            while (true) {
                const bool r0 = (unsigned)(p0 >> 32) == fin && (unsigned)(p1 >> 32) == fin &&
                                (unsigned)(p2 >> 32) == fin && (unsigned)(p3 >> 32) == fin;
                const bool r1 = (unsigned)(q0 >> 32) == fin && (unsigned)(q1 >> 32) == fin &&
                                (unsigned)(q2 >> 32) == fin && (unsigned)(q3 >> 32) == fin;
                if (r0 && r1) break;
                const unsigned long long now = gtimer();
                if (!t0) t0 = now;
                else if (now - t0 > timeout_ns) return false;
                if ((++spins & 63) == 0 && *(const volatile int*)status != 0) return false;
                if (!r0) {
                    ll_load2(a + 32 * i, p0, p1);
                    ll_load2(a + 32 * i + 16, p2, p3);
                }
                if (!r1) {
                    ll_load2(a + 32 * j1, q0, q1);
                    ll_load2(a + 32 * j1 + 16, q2, q3);
                }
            }
            va0 = make_uint4((unsigned)p0, (unsigned)p1, (unsigned)p2, (unsigned)p3);
            va1 = make_uint4((unsigned)q0, (unsigned)q1, (unsigned)q2, (unsigned)q3);
        } else {
            va0 = vload(a16 + i, as);
            va1 = vload(a16 + j1, as);
            if (RED) {
                vb0 = vload(b16 + i, bs);
                vb1 = vload(b16 + j1, bs);
            }
        }
        const uint4 r0 = RED ? vadd<DT>(va0, vb0) : va0;
        if (o1_ll) ll_store_vec(o1, i, r0, fout);
        else vstore(reinterpret_cast<uint4*>(o1) + i, r0, o1s);
        if (o2) {
            if (o2_ll) ll_store_vec(o2, i, r0, fout);
            else vstore(reinterpret_cast<uint4*>(o2) + i, r0, false);
        }
        if (i + T < nv) {
            const uint4 r1 = RED ? vadd<DT>(va1, vb1) : va1;
            if (o1_ll) ll_store_vec(o1, i + T, r1, fout);
            else vstore(reinterpret_cast<uint4*>(o1) + i + T, r1, o1s);
            if (o2) {
                if (o2_ll) ll_store_vec(o2, i + T, r1, fout);
                else vstore(reinterpret_cast<uint4*>(o2) + i + T, r1, false);
            }
        }
    }
    return true;
}

// The same with U vectors per thread in flight (the sequential engine, whose
// threads all move data): every load of a round -- LL lines and plain
// operands -- is issued before the first poll, and only the lines that do
// not carry the flag yet are read again, so a round costs one round trip
// once the producer's lines have landed.
template <bool RED, int DT, int U>
__device__ __forceinline__ bool move_ll_wide(const SlotOp& op, int tid, int T, unsigned long long timeout_ns,
                                             const int* status)
{
    constexpr int ES = (DT == CCL_BF16 || DT == CCL_F16) ? 2 : 4;
    const long long nv = op.n * ES / 16;
    const char* a = op.a;
    const uint4* a16 = reinterpret_cast<const uint4*>(a);
    const uint4* b16 = reinterpret_cast<const uint4*>(op.b);
    const bool a_ll = op.a_ll, o1_ll = op.o1_ll, o2_ll = op.o2_ll, as = op.as, bs = op.bs, o1s = op.o1s;
    char* o1 = op.o1;
    char* o2 = op.o2;
    const unsigned fin = op.fin, fout = op.fout;
    for (long long i0 = tid; i0 < nv; i0 += (long long)U * T) {
        unsigned long long x0[U], x1[U], x2[U], x3[U];
        uint4 vb[U];
        unsigned pend = 0;   // bit u: vector u of the round still lacks the slot's flag
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long j = i0 + (long long)u * T < nv ? i0 + (long long)u * T : nv - 1;
            if (a_ll) {
                ll_load2(a + 32 * j, x0[u], x1[u]);
                ll_load2(a + 32 * j + 16, x2[u], x3[u]);
            } else {
                const uint4 v = vload(a16 + j, as);
                x0[u] = v.x;
                x1[u] = v.y;
                x2[u] = v.z;
                x3[u] = v.w;
            }
            vb[u] = RED ? vload(b16 + j, bs) : make_uint4(0, 0, 0, 0);
        }
        if (a_ll) {
            unsigned long long t0 = 0;
            unsigned spins = 0;
            while (true) {
                pend = 0;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const bool ready = (unsigned)(x0[u] >> 32) == fin && (unsigned)(x1[u] >> 32) == fin &&
                                       (unsigned)(x2[u] >> 32) == fin && (unsigned)(x3[u] >> 32) == fin;
                    if (!ready && i0 + (long long)u * T < nv) pend |= 1u << u;
                }
                if (!pend) break;
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (pend & (1u << u)) {
                        const long long j = i0 + (long long)u * T;
                        ll_load2(a + 32 * j, x0[u], x1[u]);
                        ll_load2(a + 32 * j + 16, x2[u], x3[u]);
                    }
                const unsigned long long now = gtimer();
                if (!t0) t0 = now;
                else if (now - t0 > timeout_ns) return false;
                if ((++spins & 63) == 0 && *(const volatile int*)status != 0) return false;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long j = i0 + (long long)u * T;
            if (j < nv) {
                const uint4 va = make_uint4((unsigned)x0[u], (unsigned)x1[u], (unsigned)x2[u], (unsigned)x3[u]);
                const uint4 r = RED ? vadd<DT>(va, vb[u]) : va;
                if (o1_ll) ll_store_vec(o1, j, r, fout);
                else vstore(reinterpret_cast<uint4*>(o1) + j, r, o1s);
                if (o2) {
                    if (o2_ll) ll_store_vec(o2, j, r, fout);
                    else vstore(reinterpret_cast<uint4*>(o2) + j, r, false);
                }
            }
        }
    }
    return true;
}

template <int DT>
__device__ __forceinline__ bool move_ll_dt(const SlotOp& op, int tid, int T, const KParams& P)
{
    return op.red ? move_ll<true, DT>(op, tid, T, P.timeout_ns, P.status)
                  : move_ll<false, DT>(op, tid, T, P.timeout_ns, P.status);
}

template <bool LL, int MAXT>
static __device__ void data_warps(const KParams& P, CtlShared* sh)
{
    constexpr int U = InFlight<MAXT>::U;
    const int tid = threadIdx.x - 96;
    const int T = blockDim.x - 96;
    const int lane = threadIdx.x & 31;
    const unsigned long long limit = 4 * P.timeout_ns;
    for (int j = 0;; ++j) {
        const int q = j % kQ;
        if (!mbar_wait(&sh->ready[q], (unsigned)((j / kQ) & 1), limit)) {
            if (lane == 0) record_timeout(P, -1, WAIT_DONE);
            return;
        }
        // the descriptor stays put until every data warp acknowledged it
        const SlotOp& op = sh->op[q];
        if (op.cmd != 0) return;
        if (LL && (op.a_ll || op.o1_ll || op.o2_ll)) {
            // after a recorded failure the tile is only acknowledged
            if (op.n > 0 && *(volatile int*)P.status == 0) {
                bool ok;
                switch (op.dtype) {
                case CCL_F32: ok = move_ll_dt<CCL_F32>(op, tid, T, P); break;
                case CCL_BF16: ok = move_ll_dt<CCL_BF16>(op, tid, T, P); break;
                case CCL_F16: ok = move_ll_dt<CCL_F16>(op, tid, T, P); break;
                default: ok = move_ll_dt<CCL_I32>(op, tid, T, P); break;
                }
                if (!ok) record_timeout(P, -1, WAIT_FULL);
            }
        } else if (!op.bulk && op.n > 0 && op.o3) {
            copy3_call(op.a, op.o1, op.o2, op.o3, op.n, (op.dtype == CCL_BF16 || op.dtype == CCL_F16) ? 2 : 4, tid, T);
        } else if (!op.bulk && op.n > 0 && op.c) {
            move_part3_call<U>(op.dtype, op.a, op.as, op.b, op.bs, op.c, op.cs, op.o1, op.o1s, op.o2, op.n, tid, T);
        } else if (!op.bulk && op.n > 0) {
            switch (op.dtype) {
            case CCL_F32: move_part<CCL_F32, U>(op.red, op.a, op.as, op.b, op.bs, op.o1, op.o1s, op.o2, op.n, tid, T); break;
            case CCL_BF16: move_part<CCL_BF16, U>(op.red, op.a, op.as, op.b, op.bs, op.o1, op.o1s, op.o2, op.n, tid, T); break;
            case CCL_F16: move_part<CCL_F16, U>(op.red, op.a, op.as, op.b, op.bs, op.o1, op.o1s, op.o2, op.n, tid, T); break;
            default: move_part<CCL_I32, U>(op.red, op.a, op.as, op.b, op.bs, op.o1, op.o1s, op.o2, op.n, tid, T); break;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->done_g[q]);
    }
}

// ----------------------------------------------------------------------
// Sequential engine: one CTA per threadblock program, no warp roles.  Thread
// 0 waits (bounded) for a step's dependency counters and, slot by slot, for
// the FIFO flags; every thread of the CTA moves the slot; after a CTA
// barrier thread 0 issues the gpu-scope release fence and posts the slot's
// flags (and, after the last slot, the step's counter).  Steps run strictly
// one after another, so a step needs no drain of an earlier one.  Fewer
// hand-offs per step than the warp-specialised pipeline, and all warps move
// data; no overlap of one step's waits with another step's data.
// ----------------------------------------------------------------------
struct SeqShared {
    DRec rec[2];              // the current step's record and the next one, arriving by cp.async
    DLink links[kSeqLinks];   // the program's first links (KParams.prog_links)
    int go;                   // thread 0's verdict on the current wait (1: the waits were met)
};

// A threadblock program of the sequential engine may run on a cluster of
// P.cluster CTAs: every CTA moves its share of each slot, and thread 0 of
// every CTA waits for the step's counters and the slot's flags itself (the
// same words; a verdict needs no hand-over between CTAs).  group_sync, after
// the data, is the barrier of all of them (a cluster barrier with release /
// acquire at cluster scope), after which the cluster's first CTA issues the
// gpu-scope fence and posts, covering every CTA's stores.  No CTA leaves
// early: after a failed wait (recorded in the status word) a CTA skips its
// data and goes on through the same barriers as the others, whose waits
// then give up at once on the recorded status -- so a cluster never waits
// at a barrier for a CTA that has left.  No CTA touches another's shared
// memory.
__device__ __forceinline__ unsigned cluster_rank()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void group_sync(const KParams& P)
{
    if (P.cluster > 1) {
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    } else {
        __syncthreads();
    }
}
__device__ __forceinline__ bool seq_leader(const KParams& P)
{
    return threadIdx.x == 0 && (P.cluster <= 1 || cluster_rank() == 0);
}

// the LL data path of a sequential step, out of line (its polling loops
// stay out of the register budget of the step's own code)
template <int DT>
__device__ __forceinline__ bool seq_move_ll_dt(const SlotOp& op, int tid, int T, const KParams& P)
{
    constexpr int UL = 4;   // vectors per thread in flight
    return op.red ? move_ll_wide<true, DT, UL>(op, tid, T, P.timeout_ns, P.status)
                  : move_ll_wide<false, DT, UL>(op, tid, T, P.timeout_ns, P.status);
}
static __device__ __noinline__ bool seq_move_ll(const SlotOp& op, int tid, int T, const KParams& P)
{
    switch (op.dtype) {
    case CCL_F32: return seq_move_ll_dt<CCL_F32>(op, tid, T, P);
    case CCL_BF16: return seq_move_ll_dt<CCL_BF16>(op, tid, T, P);
    case CCL_F16: return seq_move_ll_dt<CCL_F16>(op, tid, T, P);
    default: return seq_move_ll_dt<CCL_I32>(op, tid, T, P);
    }
}

// Hint the lines of [p, p + bytes) into L2, one 128-byte line per thread
// and round (addresses stay inside the range)
__device__ __forceinline__ void prefetch_l2(const char* p, long long bytes, int tid, int T)
{
    if (!p) return;
    for (long long off = (long long)tid * 128; off < bytes; off += (long long)T * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p + off));
}

// One step, run by every thread of the CTA (of every CTA of the program's
// cluster) with the same record (the library's kernel reads it from shared
// memory, a generated kernel builds it from constants).  Lin / Lout: its
// links, or null.  deps / ndeps: dependency counters thread 0 waits for
// before the first slot, just before that slot's flags (null when the
// caller has waited already; pre_ok is then thread 0's verdict on that
// wait).  `go` is the CTA's shared verdict word; t_start and waited are
// thread 0's stamps for the timeline.  Never leaves early: a failed wait
// skips the CTA's data and posts (the status word holds the failure).
//
// While the leader waits, every thread hints its share of the operands that
// are not FIFO slots (the source and local buffers) into L2, so the data
// phase after the wait reads them from L2.  With the LL protocol the
// incoming slot's flag is not waited for: the threads poll the slot's lines
// themselves (move_ll), and the outgoing slot gets lines instead of a full
// flag, so no fence and flag round trip sits between two hops of a chain.
template <int U>
__device__ __forceinline__ void seq_step(const KParams& P, int* go, const DRec& st, const DLink* Lin,
                                         const DLink* Lout, const DDep* deps, int ndeps, bool pre_ok, int si,
                                         unsigned exec_mod, unsigned long long t_start, unsigned long long waited)
{
    const int C = P.cluster > 1 ? P.cluster : 1;
    const int tid = threadIdx.x, T = blockDim.x;
    const int crank = C > 1 ? (int)cluster_rank() : 0;
    const bool leader = tid == 0 && crank == 0;
    const unsigned S = (unsigned)P.S;
    const int es = (st.dtype == CCL_BF16 || st.dtype == CCL_F16) ? 2 : 4;
    const int esh = es == 2 ? 1 : 2;
    const long long ve = 16 / es;
    const long long lls = P.ll ? 2 : 1;   // slot bytes per data byte
    const unsigned long long base_in = Lin ? (unsigned long long)(P.exec * Lin->total) : 0;
    const unsigned long long base_out = Lout ? (unsigned long long)(P.exec * Lout->total) : 0;
    const long long slot_elems = P.slot_bytes >> esh;
    const bool linked = Lin || Lout;
    long long nslots = linked ? (st.nslots > 0 ? st.nslots : 1) : 1;
    if (!linked && st.nelem > 0) nslots = (st.nelem + slot_elems - 1) / slot_elems;
    unsigned in_idx = Lin ? slot_index(exec_mod, *Lin, st.seq_in_mod, S) : 0;
    unsigned out_idx = Lout ? slot_index(exec_mod, *Lout, st.seq_out_mod, S) : 0;
    const int red = kind_reduces(st.kind);
    const bool three = kind_three(st.kind);
    const char* srcb = st.src_buf >= 0 ? P.bufs[st.src_buf][st.src_rank] + st.src_off * es : nullptr;
    const char* locb = st.loc_buf >= 0 ? P.bufs[st.loc_buf][st.loc_rank] + st.loc_off * es : nullptr;
    char* dstb = st.dst_buf >= 0 ? P.bufs[st.dst_buf][st.dst_rank] + st.dst_off * es : nullptr;
    const bool a_slot = Lin && st.kind != CCL_I_REDUCE;   // the first operand is the incoming slot
    const bool post = !(st.flags & STEP_NOPOST);
    unsigned long long t_pub = 0, t_done = 0;
    for (long long k = 0; k < nslots; ++k) {
        const unsigned long long sin = base_in + st.seq_in + k;
        const unsigned long long sout = base_out + st.seq_out + k;
        long long e0 = k * slot_elems;
        long long n = st.nelem - e0;
        if (n > slot_elems) n = slot_elems;
        if (n < 0) n = 0;
        long long soff = 0;   // this CTA's share of the slot (16-byte units)
        if (C > 1) {
            const long long V = n / ve;
            const long long lo = (V * crank / C) * ve;
            const long long hi = crank == C - 1 ? n : (V * (crank + 1) / C) * ve;
            soff = lo;
            e0 += lo;
            n = hi - lo;
        }
        const char* a = (a_slot || !srcb) ? nullptr : srcb + e0 * es;
        // a two-destination copy keeps its second destination in the
        // local-operand range
        // (a folded recv-reduce-copy-send: in its source range)
        const bool copy2 = st.kind == CCL_I_COPY2 || st.kind == CCL_I_COPY3, rrc2 = st.kind == CCL_I_RRC2;
        const char* b = locb && !copy2 ? locb + e0 * es : nullptr;
        if (n > 0) {
            prefetch_l2(a, n * es, tid, T);
            prefetch_l2(b, n * es, tid, T);
            // a folded reduction chain's third operand: its source range
            if (three) prefetch_l2(srcb + e0 * es, n * es, tid, T);
        }
        if (linked || k == 0) {
            if (tid == 0) {
                int ok = k == 0 ? pre_ok : 1;
                if (k == 0 && ok && ndeps > 0) ok = wait_deps(P, deps, ndeps, si, waited, true);
                if (ok && linked)
                    ok = wait_slots(P, Lin, Lout, sin, sout, st.seq_out + k, in_idx, out_idx, 1, si, waited, true) != 0;
                *go = ok;
            }
            __syncthreads();
        }
        // this CTA's verdict (written before the barrier above; the next
        // write follows the group barrier below, which every thread reaches
        // after this read)
        const bool ok = *(volatile int*)go != 0;
        if (leader && P.timeline && k == 0) t_pub = gtimer();
        const char* slot_in = Lin ? P.fifo + Lin->slot_base + (long long)in_idx * P.slot_stride + lls * soff * es : nullptr;
        char* slot_out = Lout ? P.fifo + Lout->slot_base + (long long)out_idx * P.slot_stride + lls * soff * es : nullptr;
        bool as = false;
        if (a_slot) {
            a = slot_in;
        } else {
            as = (st.flags & STEP_SRC_STREAM) && P.stream_in;
        }
        const bool bs = (st.flags & STEP_LOC_STREAM) && P.stream_in;
        char* o1;
        char* o2 = nullptr;
        bool o1s = false;
        if (dstb) {
            o1 = dstb + e0 * es;
            o1s = st.dst_buf == CCL_BUF_OUT;
            // (a second destination -- a folded receive -- is written
            // instead of a slot; its address is made here, not kept live)
            o2 = copy2  ? const_cast<char*>(locb) + e0 * es
                 : rrc2 ? const_cast<char*>(srcb) + e0 * es
                 : st.x_buf >= 0 ? P.bufs[st.x_buf][st.x_rank] + (st.x_off + e0) * es
                                 : slot_out;
        } else {
            o1 = slot_out;
        }
        if (ok && n > 0) {
            if (P.ll && (a_slot || slot_out)) {
                SlotOp op;
                op.a = a;
                op.b = b;
                op.c = nullptr;   // no folded reduction chains with LL slots
                op.cs = 0;
                op.o3 = nullptr;
                op.o1 = o1;
                op.o2 = o2;
                op.n = n;
                op.red = red;
                op.dtype = st.dtype;
                op.as = as;
                op.bs = bs;
                op.o1s = o1s;
                op.bulk = 0;
                op.cmd = 0;
                op.a_ll = a_slot;
                op.o1_ll = !dstb;
                op.o2_ll = dstb && slot_out;
                op.fin = (unsigned)(sin + 1);
                op.fout = (unsigned)(sout + 1);
                // after a recorded failure the part is skipped; the leader
                // sees the status before its next wait
                if (*(volatile int*)P.status == 0 && !seq_move_ll(op, tid, T, P)) record_timeout(P, si, WAIT_FULL);
            } else if (st.kind == CCL_I_COPY3) {
                copy3_part(a, o1, o2, P.bufs[st.x_buf][st.x_rank] + (st.x_off + e0) * es, n, es, tid, T);
            } else if (three) {
                move_part3<U>(st.dtype, a, as, b, bs, srcb + e0 * es, (st.flags & STEP_SRC_STREAM) && P.stream_in, o1,
                              o1s, o2, n, tid, T);
            } else {
                switch (st.dtype) {
                case CCL_F32: move_part<CCL_F32, U>(red, a, as, b, bs, o1, o1s, o2, n, tid, T); break;
                case CCL_BF16: move_part<CCL_BF16, U>(red, a, as, b, bs, o1, o1s, o2, n, tid, T); break;
                case CCL_F16: move_part<CCL_F16, U>(red, a, as, b, bs, o1, o1s, o2, n, tid, T); break;
                default: move_part<CCL_I32, U>(red, a, as, b, bs, o1, o1s, o2, n, tid, T); break;
                }
            }
        }
        group_sync(P);
        if (leader) {
            if (P.timeline && k == nslots - 1) t_done = gtimer();
            // every thread's stores were observed at the barrier; the
            // fence makes them visible at gpu scope before the flags.  After
            // a failed wait (or an LL part that gave up) nothing is posted.
            // a consumed flag matters only to a producer that reuses the slot
            // within this execution; an LL slot needs no full flag; with
            // nothing to post there is no fence either (and an LL part's
            // failure needs no check)
            bool p_in = Lin && post && ok && st.seq_in + k + S < Lin->total;
            bool p_out = Lout && post && ok && !P.ll;
            bool p_sig = k == nslots - 1 && st.signal >= 0 && post && ok;
            if (P.ll && (p_in || p_sig) && *(volatile int*)P.status != 0) p_in = p_out = p_sig = false;
            // one word: a release store; several: one fence, then relaxed stores
            const bool one = (int)p_in + (int)p_out + (int)p_sig == 1;
            if ((p_in || p_out || p_sig) && !one) fence_acq_rel_gpu();
            if (p_in) post_word(P.flags + Lin->flag_base + S + in_idx, sin + 1, one);
            if (p_out) post_word(P.flags + Lout->flag_base + out_idx, sout + 1, one);
            if (k == nslots - 1) {
                if (p_sig) post_word(P.counters + st.signal, (unsigned long long)(P.exec * P.m + st.mb + 1), one);
                if (P.timeline) {
                    unsigned long long* tl = P.timeline + 5ll * si;
                    tl[0] = t_start;
                    tl[1] = waited;
                    tl[2] = t_pub;
                    tl[3] = t_done;
                    tl[4] = gtimer();
                }
            }
        }
        if (++in_idx == S) in_idx = 0;
        if (++out_idx == S) out_idx = 0;
    }
}


// mbarriers of a pipelined-engine CTA (thread 0), before the roles start
__device__ __forceinline__ void ctl_init(const KParams& P, CtlShared* sh)
{
    load_prog_links(P, blockIdx.x, sh->links);
    if (threadIdx.x == 0) {
        const int nwarps = blockDim.x / 32;
        for (int q = 0; q < kQ; ++q) {
            mbar_init(&sh->ready[q], 1);
            mbar_init(&sh->done_g[q], nwarps - 3);
            mbar_init(&sh->done_b[q], 1);
            mbar_init(&sh->freed[q], 1);
        }
        for (int s = 0; s < kNSMax; ++s) mbar_init(&sh->full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
}

// ----------------------------------------------------------------------
// Building blocks of the kernels generated for single plans (ReSCCL report,
// §II.2: one kernel per schedule instead of an instruction interpreter).
// A generated kernel walks each threadblock program as code: the constants
// of every instruction (kind, type, buffers, offsets, links, counters) are
// written into it, micro-batch pieces and FIFO sequence numbers are computed
// in loops, and each step runs the same seq_step / issue_step as the
// library's kernels -- so no step record, link or dependency table is read
// from memory.
// ----------------------------------------------------------------------

// a step with its links written out (links absent: link_in / link_out < 0)
struct GenStep {
    DRec st;
    DLink lin, lout;
};

// What every step of one channel instruction of a generated threadblock
// program shares: its record fields (offsets of the whole channel range),
// links, dependency counters and drain rule.  The generated code fills one
// per instruction, in the threadblock's own code.
struct GenInstr {
    DRec st;
    DLink lin, lout;
    int dep_first, ndep;        // its dependency counters: entries of the module's dependency list, each
                                // {counter, mode}; mode bit 0: waited at every piece with value mb + 1,
                                // bit 1: waited at piece 0 with value m
    int drain_kind;             // 0 none, 2 fixed step, 3 fixed distance back, 4 same piece of another instruction
    int drain_dk, drain_const;
    long long p_base;           // drain_kind 4: that instruction's segment (first step, instructions,
    int p_n, p_w, p_pos;        //   window) and position in it
    int qin, qout;              // the threadblock's running sequence counters of its links (-1: none)
};

// wait (bounded) for an instruction's dependency counters at piece mb, up
// to kDepBatch of them per polling round
__device__ __forceinline__ bool wait_gen_deps(const KParams& P, const GenInstr& gi, const int2* dep, int mb, int m,
                                              int si, unsigned long long& waited)
{
    DDep d[kDepBatch];
    int nd = 0;
    for (int k = 0; k < gi.ndep; ++k) {
        const int2 e = dep[gi.dep_first + k];
        if ((e.y & 1) || ((e.y & 2) && mb == 0)) {
            d[nd].counter = e.x;
            d[nd].pad = 0;
            d[nd].value = (e.y & 2) && mb == 0 ? (long long)m : (long long)mb + 1;
            if (++nd == kDepBatch) {
                if (!wait_deps(P, d, nd, si, waited)) return false;
                nd = 0;
            }
        }
    }
    return nd == 0 || wait_deps(P, d, nd, si, waited);
}

// piece k of n elements split into `parts` 16-byte-granular pieces; the
// element tail goes to the last piece (the planner's split)
__device__ __forceinline__ void gen_split(long long n, long long ve, long long parts, long long k, long long& off,
                                          long long& len)
{
    const long long V = n / ve;
    const long long a = (V * k / parts) * ve;
    const long long b = (k == parts - 1) ? n : (V * (k + 1) / parts) * ve;
    off = a;
    len = b - a;
}

// step index of micro-batch mb of the instruction at position pos of a
// segment that starts at step base and runs n instructions in windows of w
__device__ __forceinline__ long long gen_seg_step(long long base, int n, int w, int pos, int mb, int m)
{
    const int w0 = mb / w * w;
    const int wl = (w0 + w < m ? w0 + w : m) - w0;
    return base + (long long)w0 * n + (long long)pos * wl + (mb - w0);
}

// The steps of one instruction for micro-batches [w0, w1): the piece of each
// (the planner's split of the instruction's st.nelem elements into m
// pieces), its FIFO slots, the sequence numbers (q: the threadblock's
// running counts on its links), counters and drain; then the step itself.
// si: the running step index.  False when a wait gave up.
__device__ __forceinline__ void gen_piece(const GenInstr& gi, int m, long long ve, long long slot_elems, int S,
                                          int mb, long long* q, GenStep& g)
{
    long long off, len;
    gen_split(gi.st.nelem, ve, m, mb, off, len);
    g.st = gi.st;
    g.lin = gi.lin;
    g.lout = gi.lout;
    g.st.src_off += off;
    g.st.loc_off += off;
    g.st.dst_off += off;
    if (g.st.x_buf >= 0) g.st.x_off += off;
    g.st.nelem = len;
    const bool linked = gi.st.link_in >= 0 || gi.st.link_out >= 0;
    const long long ns = (len + slot_elems - 1) / slot_elems;
    g.st.nslots = linked ? (int)(ns > 1 ? ns : 1) : 0;
    if (gi.st.link_in >= 0) {
        long long& qin = q[gi.qin];
        g.st.seq_in = qin;
        g.st.seq_in_mod = (int)(qin % S);
        qin += g.st.nslots;
    }
    if (gi.st.link_out >= 0) {
        long long& qout = q[gi.qout];
        g.st.seq_out = qout;
        g.st.seq_out_mod = (int)(qout % S);
        qout += g.st.nslots;
    }
    g.st.mb = mb;
}

// sequential engine: thread 0 of every CTA writes the piece's step into
// the CTA's shared `gs` (and keeps the link counters q) and waits for its
// counters, then the CTA (the cluster) runs it.  Always true: a failed wait
// leaves the failure in the status word and the program runs on without
// data (see seq_step).
template <int U>
__device__ __noinline__ bool gen_seq_block(const KParams& P, int* go, GenStep* gs, const GenInstr& gi,
                                           const int2* dep, int w0, int w1, int m, long long ve,
                                           long long slot_elems, int S, int& si, long long* q, unsigned exec_mod)
{
#pragma unroll 1
    for (int mb = w0; mb < w1; ++mb, ++si) {
        unsigned long long t_start = 0, waited = 0;
        bool ok = true;
        if (threadIdx.x == 0) {
            gen_piece(gi, m, ve, slot_elems, S, mb, q, *gs);
            gs->st.drain = -1;
            if (P.timeline) t_start = gtimer();
            if (gi.ndep > 0) ok = wait_gen_deps(P, gi, dep, mb, m, si, waited);
        }
        __syncthreads();   // gs holds the piece
        seq_step<U>(P, go, gs->st, gs->st.link_in >= 0 ? &gs->lin : nullptr,
                    gs->st.link_out >= 0 ? &gs->lout : nullptr, nullptr, 0, ok, si, exec_mod, t_start, waited);
        __syncthreads();   // gs takes the next piece
    }
    return true;
}

// Poll, in one round trip of relaxed loads, the first-slot flags and the
// first kDepPoll dependency counters of pieces g[0..n) of one instruction;
// the length (>= 1) of the leading run whose words are all ready, after one
// acquire fence, or 0 when the wait for g[0] fails.
__device__ __forceinline__ int gen_poll(const KParams& P, const GenStep* g, int n, const GenInstr& gi,
                                        const int2* dep, int m, unsigned exec_mod, int si,
                                        unsigned long long& waited)
{
    constexpr int kC = 2 + kDepPoll;
    const unsigned long long* ptr[kLook * kC];
    unsigned long long want[kLook * kC];
    const unsigned long long base = (unsigned long long)(P.exec * P.m);
#pragma unroll
    for (int i = 0; i < kLook; ++i) {
        for (int k = 0; k < kC; ++k) ptr[i * kC + k] = nullptr;
        if (i >= n) continue;
        const SlotCond c = first_slot_cond(P, g[i].st, exec_mod, g[i].st.link_in >= 0 ? &g[i].lin : nullptr,
                                           g[i].st.link_out >= 0 ? &g[i].lout : nullptr);
        ptr[i * kC] = c.in;
        want[i * kC] = c.vin;
        ptr[i * kC + 1] = c.out;
        want[i * kC + 1] = c.vout;
        int k = 0;
        for (int e = 0; e < gi.ndep && k < kDepPoll; ++e) {
            const int2 d = dep[gi.dep_first + e];
            const int mb = g[i].st.mb;
            if ((d.y & 1) || ((d.y & 2) && mb == 0)) {
                ptr[i * kC + 2 + k] = P.counters + d.x;
                want[i * kC + 2 + k] = base + ((d.y & 2) && mb == 0 ? (unsigned long long)m : (unsigned long long)mb + 1);
                ++k;
            }
        }
    }
    unsigned long long t0 = 0;
    unsigned spins = 0;
    while (true) {
        unsigned long long x[kLook * kC];
#pragma unroll
        for (int k = 0; k < kLook * kC; ++k) x[k] = ptr[k] ? ld_relaxed(ptr[k]) : ~0ull;
        int r = 0;
        bool ok = true;
#pragma unroll
        for (int i = 0; i < kLook; ++i) {
#pragma unroll
            for (int k = 0; k < kC; ++k)
                if (ptr[i * kC + k] && x[i * kC + k] < want[i * kC + k]) ok = false;
            if (ok && i < n) r = i + 1;
        }
        if (r > 0) {
            fence_acq_rel_gpu();
            if (t0) waited += gtimer() - t0;
            return r;
        }
        if (!t0) t0 = gtimer();
        ++spins;
        if ((spins & 15) == 0) {
            if (*(volatile int*)P.status != 0) return 0;
            if (gtimer() - t0 > P.timeout_ns) {
                record_timeout(P, si, ptr[0] && x[0] < want[0] ? WAIT_FULL : ptr[1] && x[1] < want[1] ? WAIT_FREE
                                                                                                    : WAIT_DEP);
                return 0;
            }
        }
        if (spins > 64) __nanosleep(32);
    }
}

// pipelined engine, issuing thread: the pieces of one instruction for
// micro-batches [w0, w1), kLook at a time: one batched poll of their first
// slots and counters, then each piece's drain and remaining counters, then
// its slots handed out
static __device__ __noinline__ bool gen_issue_block(const KParams& P, CtlShared* sh, const GenInstr& gi,
                                                    const int2* dep, int w0, int w1, int m, long long ve,
                                                    long long slot_elems, int S, int& si, int& head, long long* q,
                                                    unsigned exec_mod)
{
    const unsigned long long limit = 4 * P.timeout_ns;
#pragma unroll 1
    for (int b0 = w0; b0 < w1; b0 += kLook) {
        const int n = w1 - b0 < kLook ? w1 - b0 : kLook;
        GenStep g[kLook];
        for (int i = 0; i < n; ++i) {
            const int mb = b0 + i;
            gen_piece(gi, m, ve, slot_elems, S, mb, q, g[i]);
            int drain = -1;
            if (gi.drain_kind == 2) drain = gi.drain_const;
            else if (gi.drain_kind == 3) drain = si + i - gi.drain_dk;
            else if (gi.drain_kind == 4) drain = (int)gen_seg_step(gi.p_base, gi.p_n, gi.p_w, gi.p_pos, mb, m);
            g[i].st.drain = drain;
        }
        int i = 0;
        while (i < n) {
            const unsigned long long t_start = gtimer();
            unsigned long long waited = 0;
            const int r = gen_poll(P, g + i, n - i, gi, dep, m, exec_mod, si, waited);
            if (r == 0) {
                publish_cmd(sh, head, 2, limit);
                return false;
            }
            for (int j = 0; j < r; ++j, ++i, ++si) {
                const GenStep& s = g[i];
                if (!wait_drain(P, sh, s.st.drain, si, head) ||
                    (gi.ndep > kDepPoll && !wait_gen_deps(P, gi, dep, s.st.mb, m, si, waited))) {
                    publish_cmd(sh, head, 2, limit);
                    return false;
                }
                if (!issue_step(P, sh, s.st, s.st.link_in >= 0 ? &s.lin : nullptr,
                                s.st.link_out >= 0 ? &s.lout : nullptr, si, head, 1, exec_mod, t_start, waited))
                    return false;
            }
        }
    }
    return true;
}

}  // namespace ccl
