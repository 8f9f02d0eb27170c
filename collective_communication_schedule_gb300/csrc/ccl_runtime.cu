// C ABI entry points, device plan management and the executor kernel.
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "ccl_device.cuh"
#include "ccl_executor.cuh"
#include "ccl_internal.h"
#include "ccl_plan.h"

// ======================================================================
// errors
// ======================================================================
namespace ccl {
static thread_local std::string g_detail;
void set_error(const std::string& msg) { g_detail = msg; }
ccl_status_t fail(ccl_status_t st, const std::string& msg)
{
    g_detail = msg;
    return st;
}
static ccl_status_t cuda_fail(cudaError_t e, const char* what)
{
    return fail(e == cudaErrorMemoryAllocation ? CCL_ERR_OOM : CCL_ERR_CUDA,
                std::string(what) + ": " + cudaGetErrorString(e));
}
}  // namespace ccl

#define CUDA_TRY(call, what)                                        \
    do {                                                            \
        cudaError_t _e = (call);                                    \
        if (_e != cudaSuccess) return ccl::cuda_fail(_e, what);     \
    } while (0)

// ======================================================================
// device code
// ======================================================================
namespace ccl {

// ----------------------------------------------------------------------
// Warp-specialised executor.  Four roles per CTA:
//
//  * issuer (warp 0, lane 0) walks the threadblock program.  Step records
//    (128 bytes each) arrive by cp.async in batches of kLook, one batch
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
    char* o1;           // destination buffer, or the outgoing slot
    char* o2;           // outgoing slot when a destination is also written
    long long n;        // elements
    int red, dtype;
    int as, bs, o1s;    // streaming cache hints (register path)
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
};

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
__device__ bool wait_deps(const KParams& P, const DDep* deps, int n, int si, unsigned long long& waited)
{
    const unsigned long long base = (unsigned long long)(P.exec * P.m);
    unsigned long long t0 = 0;
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
// wait for the first one fails.
constexpr int kBatch = 4;
__device__ int wait_slots(const KParams& P, const DLink* Lin, const DLink* Lout, unsigned long long sin0,
                          unsigned long long sout0, unsigned in_idx0, unsigned out_idx0, int bmax, int si,
                          unsigned long long& waited)
{
    const unsigned S = (unsigned)P.S;
    unsigned long long t0 = 0;
    unsigned spins = 0;
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
                if (Lin && !P.ll) x[i] = ld_relaxed(P.flags + Lin->flag_base + ii);
                if (Lout && sout0 + i + 1 > (unsigned long long)P.S) y[i] = ld_relaxed(P.flags + Lout->flag_base + S + io);
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
    for (int k = 0; k < 8; ++k)
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

__device__ __forceinline__ SlotCond first_slot_cond(const KParams& P, const DRec& st, unsigned exec_mod)
{
    SlotCond c{nullptr, nullptr, 0, 0};
    const unsigned S = (unsigned)P.S;
    if (st.link_in >= 0 && !P.ll) {   // LL: the data path polls the lines
        const DLink& L = P.links[st.link_in];
        const unsigned long long s = (unsigned long long)(P.exec * L.total) + st.seq_in;
        c.in = P.flags + L.flag_base + slot_index(exec_mod, L, st.seq_in_mod, S);
        c.vin = s + 1;
    }
    if (st.link_out >= 0) {
        const DLink& L = P.links[st.link_out];
        const unsigned long long s = (unsigned long long)(P.exec * L.total) + st.seq_out;
        if (s + 1 > (unsigned long long)P.S) {
            c.out = P.flags + L.flag_base + S + slot_index(exec_mod, L, st.seq_out_mod, S);
            c.vout = s + 1 - P.S;
        }
    }
    return c;
}

// Poll the conditions of steps [s0, s1) (records in the ring) -- the first
// FIFO slot's flags and the first kDepPoll dependency counters of each --
// with relaxed loads issued together; returns the end of the leading run of
// ready steps (> s0) after one acquire fence, or -1 when the wait for step
// s0 fails.  Counters of a step beyond kDepPoll are left to wait_deps.
__device__ int poll_steps(const KParams& P, CtlShared* sh, int s0, int s1, unsigned exec_mod,
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
        const SlotCond c = first_slot_cond(P, st, exec_mod);
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

__device__ __forceinline__ bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

__device__ void issuer(const KParams& P, CtlShared* sh, int b0, int b1)
{
    int head = 0;
    const unsigned long long limit = 4 * P.timeout_ns;
    auto publish_cmd = [&](int cmd) {
        const int q = head % kQ;
        if (head >= kQ) mbar_wait(&sh->freed[q], (unsigned)(((head / kQ) - 1) & 1), limit);
        sh->op[q].cmd = cmd;
        mbar_arrive(&sh->ready[q]);
    };
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
    const unsigned S = (unsigned)P.S;
    const unsigned exec_mod = (unsigned)(P.exec % P.S);
    for (int si = b0; si < b1; ++si) {
        if (si >= rec_ready) {
            asm volatile("cp.async.wait_all;" ::: "memory");
            rec_ready = rec_end;
            if (rec_end < b1) request(rec_end);
        }
        const DRec& st = sh->rec[si % (2 * kLook)];
        const unsigned long long t_start = gtimer();
        unsigned long long waited = 0, t_pub = 0;
        if (si >= cleared) {
            // one round trip for the first-slot flags and dependency
            // counters of the next steps whose records are here
            const int s1 = rec_ready < si + kLook ? rec_ready : si + kLook;
            cleared = poll_steps(P, sh, si, s1, exec_mod, waited);
            if (cleared < 0) {
                publish_cmd(2);
                return;
            }
        }
        if (st.drain >= 0 && si - st.drain < kHist) {
            // reads or writes what an earlier step of this threadblock
            // touched: that step's last tile (and so, freed in order, all of
            // its tiles) must be finished first
            const int h = sh->last_head[st.drain % kHist];
            if (h >= head - kQ && !mbar_wait(&sh->freed[h % kQ], (unsigned)((h / kQ) & 1), limit)) {
                record_timeout(P, si, WAIT_DONE);
                publish_cmd(2);
                return;
            }
        }
        if (st.dep_count > kDepPoll &&
            !wait_deps(P, P.deps + st.dep_begin + kDepPoll, st.dep_count - kDepPoll, si, waited)) {
            publish_cmd(2);
            return;
        }
        const int es = (st.dtype == CCL_BF16 || st.dtype == CCL_F16) ? 2 : 4;
        const DLink* Lin = st.link_in >= 0 ? P.links + st.link_in : nullptr;
        const DLink* Lout = st.link_out >= 0 ? P.links + st.link_out : nullptr;
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
        const int red = st.kind == CCL_I_REDUCE || st.kind == CCL_I_RRC || st.kind == CCL_I_RRS || st.kind == CCL_I_RRCS;
        const char* srcb = st.src_buf >= 0 ? P.bufs[st.src_buf][st.src_rank] + st.src_off * es : nullptr;
        const char* locb = st.loc_buf >= 0 ? P.bufs[st.loc_buf][st.loc_rank] + st.loc_off * es : nullptr;
        char* dstb = st.dst_buf >= 0 ? P.bufs[st.dst_buf][st.dst_rank] + st.dst_off * es : nullptr;
        const bool post = !(st.flags & STEP_NOPOST);
        int ready_slots = si < cleared ? 1 : 0;   // slots whose flags were already seen ready
        for (long long k = 0; k < nslots; ++k) {
            const unsigned long long sin = base_in + st.seq_in + k;
            const unsigned long long sout = base_out + st.seq_out + k;
            if (linked && ready_slots == 0) {
                const int bmax = (int)((nslots - k) < kBatch ? (nslots - k) : kBatch);
                ready_slots = wait_slots(P, Lin, Lout, sin, sout, in_idx, out_idx, bmax, si, waited);
                if (ready_slots == 0) {
                    publish_cmd(2);
                    return;
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
                    publish_cmd(2);
                    return;
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
                op.b = locb ? locb + off : nullptr;
                op.bs = (st.flags & STEP_LOC_STREAM) && P.stream_in;
                if (dstb) {
                    op.o1 = dstb + off;
                    op.o1s = st.dst_buf == CCL_BUF_OUT;
                    op.o2 = slot_out ? slot_out + lls * soff : nullptr;
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
                op.bulk = P.ns > 0 && !red && tn > 0 && ((tn * es) & 15) == 0 && aligned16(op.a) &&
                          aligned16(op.o1) && (!op.o2 || aligned16(op.o2)) && !op.a_ll && !op.o1_ll && !op.o2_ll;
                op.cmd = 0;
                Release& r = sh->rel[q];
                const bool last_tile = u == ntiles - 1;
                r.consumed = (Lin && post && last_tile) ? P.flags + Lin->flag_base + S + in_idx : nullptr;
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
    }
    publish_cmd(1);
}

__device__ void releaser(const KParams& P, CtlShared* sh)
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
__device__ void tma_thread(const KParams& P, CtlShared* sh, unsigned char* stages)
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

template <int DT>
__device__ __forceinline__ bool move_ll_dt(const SlotOp& op, int tid, int T, const KParams& P)
{
    return op.red ? move_ll<true, DT>(op, tid, T, P.timeout_ns, P.status)
                  : move_ll<false, DT>(op, tid, T, P.timeout_ns, P.status);
}

template <bool LL>
__device__ void data_warps(const KParams& P, CtlShared* sh)
{
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
        } else if (!op.bulk && op.n > 0) {
            switch (op.dtype) {
            case CCL_F32: move_part<CCL_F32>(op.red, op.a, op.as, op.b, op.bs, op.o1, op.o1s, op.o2, op.n, tid, T); break;
            case CCL_BF16: move_part<CCL_BF16>(op.red, op.a, op.as, op.b, op.bs, op.o1, op.o1s, op.o2, op.n, tid, T); break;
            case CCL_F16: move_part<CCL_F16>(op.red, op.a, op.as, op.b, op.bs, op.o1, op.o1s, op.o2, op.n, tid, T); break;
            default: move_part<CCL_I32>(op.red, op.a, op.as, op.b, op.bs, op.o1, op.o1s, op.o2, op.n, tid, T); break;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->done_g[q]);
    }
}

// one instantiation per FIFO protocol: only plans with LL slots carry the
// LL data path; they run without the bulk path, with at most 512 threads
// and so twice the registers per thread
constexpr int kMaxThreadsLL = 512;
template <bool LL>
__global__ void __launch_bounds__(LL ? kMaxThreadsLL : 1024, 1) ccl_exec_kernel(const __grid_constant__ KParams P)
{
    __shared__ __align__(16) CtlShared sh;
    extern __shared__ __align__(128) unsigned char stages[];
    const int b0 = P.tb_begin[blockIdx.x], b1 = P.tb_begin[blockIdx.x + 1];
    const int nwarps = blockDim.x / 32;
    if (threadIdx.x == 0) {
        for (int q = 0; q < kQ; ++q) {
            mbar_init(&sh.ready[q], 1);
            mbar_init(&sh.done_g[q], nwarps - 3);
            mbar_init(&sh.done_b[q], 1);
            mbar_init(&sh.freed[q], 1);
        }
        for (int s = 0; s < kNSMax; ++s) mbar_init(&sh.full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    if (warp < 3) {
        if ((threadIdx.x & 31) == 0) {
            if (warp == 0) issuer(P, &sh, b0, b1);
            else if (warp == 1) releaser(P, &sh);
            else tma_thread(P, &sh, stages);
        }
        return;
    }
    data_warps<LL>(P, &sh);
}

template __global__ void ccl_exec_kernel<false>(const __grid_constant__ KParams P);
template __global__ void ccl_exec_kernel<true>(const __grid_constant__ KParams P);

// ----------------------------------------------------------------------
// Sequential engine: one CTA per threadblock program, no warp roles.  Thread
// 0 reads a step's record, waits (bounded) for its dependency counters and,
// slot by slot, for the FIFO flags; every thread of the CTA moves the slot;
// after a CTA barrier thread 0 issues the gpu-scope release fence and posts
// the slot's flags (and, after the last slot, the step's counter).  Steps run
// strictly one after another, so a step needs no drain of an earlier one.
// Fewer hand-offs per step than the warp-specialised pipeline, and all warps
// move data; no overlap of one step's waits with another step's data.
// ----------------------------------------------------------------------
struct SeqShared {
    DRec rec;
    int abort;
};

__global__ void __launch_bounds__(1024, 1) ccl_exec_seq_kernel(const __grid_constant__ KParams P)
{
    __shared__ __align__(16) SeqShared sh;
    const int tid = threadIdx.x, T = blockDim.x;
    const int b0 = P.tb_begin[blockIdx.x], b1 = P.tb_begin[blockIdx.x + 1];
    const unsigned S = (unsigned)P.S;
    const unsigned exec_mod = (unsigned)(P.exec % P.S);
    const DRec& st = sh.rec;
    for (int si = b0; si < b1; ++si) {
        unsigned long long t_start = 0, waited = 0;
        if (tid == 0) {
            if (P.timeline) t_start = gtimer();
            sh.rec = P.recs[si];
            int ok = *(volatile int*)P.status == 0;
            if (ok && sh.rec.dep_count > 0)
                ok = wait_deps(P, P.deps + sh.rec.dep_begin, sh.rec.dep_count, si, waited);
            sh.abort = !ok;
        }
        __syncthreads();
        if (sh.abort) return;
        const int es = (st.dtype == CCL_BF16 || st.dtype == CCL_F16) ? 2 : 4;
        const int esh = es == 2 ? 1 : 2;
        const DLink* Lin = st.link_in >= 0 ? P.links + st.link_in : nullptr;
        const DLink* Lout = st.link_out >= 0 ? P.links + st.link_out : nullptr;
        const unsigned long long base_in = Lin ? (unsigned long long)(P.exec * Lin->total) : 0;
        const unsigned long long base_out = Lout ? (unsigned long long)(P.exec * Lout->total) : 0;
        const long long slot_elems = P.slot_bytes >> esh;
        const bool linked = Lin || Lout;
        long long nslots = linked ? (st.nslots > 0 ? st.nslots : 1) : 1;
        if (!linked && st.nelem > 0) nslots = (st.nelem + slot_elems - 1) / slot_elems;
        unsigned in_idx = Lin ? slot_index(exec_mod, *Lin, st.seq_in_mod, S) : 0;
        unsigned out_idx = Lout ? slot_index(exec_mod, *Lout, st.seq_out_mod, S) : 0;
        const int red = st.kind == CCL_I_REDUCE || st.kind == CCL_I_RRC || st.kind == CCL_I_RRS || st.kind == CCL_I_RRCS;
        const char* srcb = st.src_buf >= 0 ? P.bufs[st.src_buf][st.src_rank] + st.src_off * es : nullptr;
        const char* locb = st.loc_buf >= 0 ? P.bufs[st.loc_buf][st.loc_rank] + st.loc_off * es : nullptr;
        char* dstb = st.dst_buf >= 0 ? P.bufs[st.dst_buf][st.dst_rank] + st.dst_off * es : nullptr;
        const bool post = !(st.flags & STEP_NOPOST);
        unsigned long long t_pub = 0, t_done = 0;
        for (long long k = 0; k < nslots; ++k) {
            const unsigned long long sin = base_in + st.seq_in + k;
            const unsigned long long sout = base_out + st.seq_out + k;
            if (linked) {
                if (tid == 0) sh.abort = wait_slots(P, Lin, Lout, sin, sout, in_idx, out_idx, 1, si, waited) == 0;
                __syncthreads();
                if (sh.abort) return;
            }
            if (tid == 0 && P.timeline && k == 0) t_pub = gtimer();
            const long long e0 = k * slot_elems;
            long long n = st.nelem - e0;
            if (n > slot_elems) n = slot_elems;
            if (n < 0) n = 0;
            const char* slot_in = Lin ? P.fifo + Lin->slot_base + (long long)in_idx * P.slot_stride : nullptr;
            char* slot_out = Lout ? P.fifo + Lout->slot_base + (long long)out_idx * P.slot_stride : nullptr;
            const char* a;
            bool as = false;
            if (Lin && st.kind != CCL_I_REDUCE) {
                a = slot_in;
            } else {
                a = srcb + e0 * es;
                as = (st.flags & STEP_SRC_STREAM) && P.stream_in;
            }
            const char* b = locb ? locb + e0 * es : nullptr;
            const bool bs = (st.flags & STEP_LOC_STREAM) && P.stream_in;
            char* o1;
            char* o2 = nullptr;
            bool o1s = false;
            if (dstb) {
                o1 = dstb + e0 * es;
                o1s = st.dst_buf == CCL_BUF_OUT;
                o2 = slot_out;
            } else {
                o1 = slot_out;
            }
            if (n > 0) {
                switch (st.dtype) {
                case CCL_F32: move_part<CCL_F32>(red, a, as, b, bs, o1, o1s, o2, n, tid, T); break;
                case CCL_BF16: move_part<CCL_BF16>(red, a, as, b, bs, o1, o1s, o2, n, tid, T); break;
                case CCL_F16: move_part<CCL_F16>(red, a, as, b, bs, o1, o1s, o2, n, tid, T); break;
                default: move_part<CCL_I32>(red, a, as, b, bs, o1, o1s, o2, n, tid, T); break;
                }
            }
            __syncthreads();
            if (tid == 0) {
                if (P.timeline && k == nslots - 1) t_done = gtimer();
                // every thread's stores were observed at the barrier; the
                // fence makes them visible at gpu scope before the flags
                fence_acq_rel_gpu();
                if (Lin && post) st_relaxed(P.flags + Lin->flag_base + S + in_idx, sin + 1);
                if (Lout && post) st_relaxed(P.flags + Lout->flag_base + out_idx, sout + 1);
                if (k == nslots - 1) {
                    if (st.signal >= 0 && post)
                        st_relaxed(P.counters + st.signal, (unsigned long long)(P.exec * P.m + st.mb + 1));
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
        __syncthreads();   // the record is read again by thread 0 for the next step
    }
}

const void* exec_kernel(int protocol, int engine)
{
    if (engine == CCL_ENGINE_SEQUENTIAL) return (const void*)ccl_exec_seq_kernel;
    return protocol == CCL_PROTO_LL ? (const void*)ccl_exec_kernel<true> : (const void*)ccl_exec_kernel<false>;
}

}  // namespace ccl

// ======================================================================
// host plan
// ======================================================================
struct ccl_plan {
    ccl::PlanImage img;
    int device = 0;
    int nranks = 0;
    char* d_blob = nullptr;
    unsigned long long* d_flags = nullptr;    // links * 2S, then counters
    char* d_fifo = nullptr;
    int* d_status = nullptr;
    unsigned long long* d_timeline = nullptr;
    char* d_scratch[CCL_MAX_RANKS] = {};
    size_t flags_count = 0;
    long long exec = 0;
    int64_t device_bytes = 0;
    double compile_ms = 0;
    ccl::KParams kp{};
    // overlapped host round trip: input copies done, kernel done, output
    // copies done (created on first use)
    cudaEvent_t ev_in = nullptr, ev_k = nullptr, ev_out = nullptr;
    bool pipe_started = false;
};

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

ccl_plan_opts_t merged_opts(const ccl_plan_opts_t* opts)
{
    ccl_plan_opts_t o;
    ccl_plan_opts_default(&o);
    o.nthreads = 512;
    if (opts) {
        if (opts->channels) o.channels = opts->channels;
        if (opts->nthreads) o.nthreads = opts->nthreads;
        if (opts->slot_bytes) o.slot_bytes = opts->slot_bytes;
        if (opts->fifo_slots) o.fifo_slots = opts->fifo_slots;
        o.microbatches = opts->microbatches;
        o.scheduler = opts->scheduler;
        o.tb_alloc = opts->tb_alloc;
        o.mb_order = opts->mb_order;
        if (opts->timeout_ms) o.timeout_ms = opts->timeout_ms;
        o.instrument = opts->instrument;
        if (opts->tile_bytes) o.tile_bytes = opts->tile_bytes;
        o.bulk = opts->bulk;
        o.link_mode = opts->link_mode;
        o.channel_scaling = opts->channel_scaling;
        o.mb_window = opts->mb_window;
        o.protocol = opts->protocol;
        o.tb_budget = opts->tb_budget;
        o.engine = opts->engine;
    }
    return o;
}

void fill_stats(const ccl::PlanImage& img, ccl_plan_stats_t* st)
{
    std::memset(st, 0, sizeof(*st));
    st->schedule_bytes = img.schedule_bytes;
    st->min_bytes = img.min_bytes;
    st->data_bytes_per_rank = img.data_bytes_per_rank;
    st->busbw_factor = img.busbw_factor;
    st->nthreadblocks = img.ntb;
    st->nthreadblocks_connection = img.ntb_connection;
    st->nsteps = (int32_t)img.steps.size();
    st->ninstr = (int32_t)img.instrs.size();
    st->nlinks = (int32_t)img.links.size();
    st->nsubpipelines = img.nsubpipelines;
    st->microbatches = img.m;
    st->mb_order = img.mb_order;
    st->channels = img.channels;
    st->nthreads = img.nthreads;
    st->fifo_slots = img.S;
    st->slot_bytes = img.slot_bytes;
    st->fifo_bytes = img.fifo_bytes;
    st->tile_bytes = img.tile_bytes;
    st->stages = img.ns;
    st->mb_window = img.mb_window;
    st->protocol = img.protocol;
    st->engine = img.engine;
    st->fuse = img.fuse;
}

void free_plan(ccl_plan* p)
{
    if (!p) return;
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(p->device);
    cudaFree(p->d_blob);
    cudaFree(p->d_flags);
    cudaFree(p->d_fifo);
    cudaFree(p->d_status);
    cudaFree(p->d_timeline);
    for (int r = 0; r < CCL_MAX_RANKS; ++r) cudaFree(p->d_scratch[r]);
    for (cudaEvent_t e : {p->ev_in, p->ev_k, p->ev_out})
        if (e) cudaEventDestroy(e);
    cudaSetDevice(prev);
    delete p;
}

ccl_status_t reset_flags(ccl_plan* p, cudaStream_t s)
{
    if (p->flags_count)
        CUDA_TRY(cudaMemsetAsync(p->d_flags, 0, p->flags_count * sizeof(unsigned long long), s), "reset flags");
    CUDA_TRY(cudaMemsetAsync(p->d_status, 0, 4 * sizeof(int), s), "reset status");
    // LL lines carry sequence numbers as well: sequences that start over
    // must not meet lines of an earlier run
    if (p->img.protocol == CCL_PROTO_LL && p->d_fifo)
        CUDA_TRY(cudaMemsetAsync(p->d_fifo, 0, p->img.fifo_bytes, s), "clear LL slots");
    p->exec = 0;
    return CCL_OK;
}

}  // namespace

extern "C" {

const char* ccl_version(void) { return "ccl-gb300 0.1 (sm_103a)"; }

const char* ccl_error_string(ccl_status_t s)
{
    switch (s) {
    case CCL_OK: return "ok";
    case CCL_ERR_INVALID_ARG: return "invalid argument";
    case CCL_ERR_CYCLE: return "dependency cycle";
    case CCL_ERR_DEADLOCK: return "deadlock";
    case CCL_ERR_RACE: return "data race";
    case CCL_ERR_UNSUPPORTED: return "unsupported";
    case CCL_ERR_OOM: return "out of device memory";
    case CCL_ERR_CUDA: return "CUDA error";
    case CCL_ERR_TIMEOUT: return "device wait timed out";
    case CCL_ERR_INTERNAL: return "internal error";
    }
    return "unknown status";
}

const char* ccl_last_error_detail(void) { return ccl::g_detail.c_str(); }

void ccl_plan_opts_default(ccl_plan_opts_t* o)
{
    if (!o) return;
    o->channels = 1;
    o->nthreads = 0;  // 0: 512, halved until all threadblocks are co-resident
    o->slot_bytes = 128 * 1024;
    o->fifo_slots = 4;
    o->microbatches = 0;
    o->scheduler = CCL_SCHED_HPDS;
    o->tb_alloc = CCL_TB_CONNECTION;
    o->mb_order = CCL_MB_AUTO;
    o->timeout_ms = 2000;
    o->instrument = 0;
    o->tile_bytes = 16 * 1024;
    o->bulk = 0;
    o->link_mode = CCL_LINK_DIRECT;
    o->channel_scaling = 1;
    o->mb_window = 0;
    o->protocol = CCL_PROTO_SIMPLE;
    o->tb_budget = 0;
    o->engine = CCL_ENGINE_PIPELINED;
}

ccl_status_t ccl_schedule_compile(const ccl_op_t* ops, int32_t nops, int32_t nranks, const int32_t nchunks[3],
                                  int32_t fuse, ccl_schedule_t* out)
{
    if (!out || !nchunks) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    auto* s = new ccl_schedule();
    ccl_status_t st = ccl::compile_program(ops, nops, nranks, nchunks,
                                           fuse == CCL_FUSE_NOCHAIN ? CCL_FUSE_NOCHAIN
                                                                    : (fuse != 0 ? CCL_FUSE_FULL : CCL_FUSE_NONE),
                                           s);
    if (st != CCL_OK) { delete s; return st; }
    *out = s;
    return CCL_OK;
}

ccl_status_t ccl_schedule_builtin(int32_t kind, int32_t nranks, int32_t group_size, uint32_t flags,
                                  ccl_schedule_t* out)
{
    if (!out) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    std::vector<ccl_op_t> ops;
    int32_t nch[3] = {0, 0, 0};
    ccl_status_t st = ccl::builtin_program(kind, nranks, group_size, flags, &ops, nch);
    if (st != CCL_OK) return st;
    auto* s = new ccl_schedule();
    st = ccl::compile_program(ops.data(), (int)ops.size(), nranks, nch, ccl::fuse_mode(flags), s);
    if (st != CCL_OK) { delete s; return st; }
    s->builtin = kind;
    s->group_size = group_size;
    *out = s;
    return CCL_OK;
}

ccl_status_t ccl_schedule_alltoallv(int32_t nranks, const int32_t* counts, uint32_t flags, ccl_schedule_t* out)
{
    if (!out) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    std::vector<ccl_op_t> ops;
    int32_t nch[3] = {0, 0, 0};
    ccl_status_t st = ccl::alltoallv_program(nranks, counts, &ops, nch);
    if (st != CCL_OK) return st;
    auto* s = new ccl_schedule();
    st = ccl::compile_program(ops.data(), (int)ops.size(), nranks, nch, ccl::fuse_mode(flags), s);
    if (st != CCL_OK) { delete s; return st; }
    s->builtin = CCL_ALLTOALLV;
    s->group_size = 0;
    *out = s;
    return CCL_OK;
}

ccl_status_t ccl_schedule_info(ccl_schedule_t s, ccl_schedule_info_t* info)
{
    if (!s || !info) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    std::memset(info, 0, sizeof(*info));
    info->nranks = s->nranks;
    for (int b = 0; b < 3; ++b) info->nchunks[b] = s->nchunks[b];
    info->nops = (int32_t)s->ops.size();
    info->ninstr = (int32_t)s->instrs.size();
    info->ntransfers = (int32_t)s->xfers.size();
    int64_t bytes = 0;
    for (const auto& I : s->instrs) {
        info->kind_count[I.kind]++;
        bytes += ccl::kind_bytes_factor(I.kind) * I.count;
    }
    info->bytes_per_chunk_elem_x_esize = bytes;
    info->builtin = s->builtin;
    info->group_size = s->group_size;
    return CCL_OK;
}

ccl_status_t ccl_schedule_get_ops(ccl_schedule_t s, ccl_op_t* ops, int32_t cap, int32_t* n)
{
    if (!s || !n) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    *n = (int32_t)s->ops.size();
    if (cap < *n || (*n && !ops)) return ccl::fail(CCL_ERR_INVALID_ARG, "capacity too small");
    std::copy(s->ops.begin(), s->ops.end(), ops);
    return CCL_OK;
}

ccl_status_t ccl_schedule_get_instrs(ccl_schedule_t s, ccl_instr_info_t* out, int32_t cap, int32_t* n)
{
    if (!s || !n) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    *n = (int32_t)s->instrs.size();
    if (cap < *n || (*n && !out)) return ccl::fail(CCL_ERR_INVALID_ARG, "capacity too small");
    for (int i = 0; i < *n; ++i) {
        const ccl::Instr& I = s->instrs[i];
        ccl_instr_info_t& o = out[i];
        o.kind = I.kind;
        o.rank = I.rank;
        o.src_rank = I.src.rank; o.src_buf = I.src.buf; o.src_off = (int32_t)I.src.off;
        o.loc_rank = I.loc.rank; o.loc_buf = I.loc.buf; o.loc_off = (int32_t)I.loc.off;
        o.dst_rank = I.dst.rank; o.dst_buf = I.dst.buf; o.dst_off = (int32_t)I.dst.off;
        o.count = (int32_t)I.count;
        o.peer_in = I.xfer_in >= 0 ? s->xfers[I.xfer_in].src_rank : -1;
        o.peer_out = I.xfer_out >= 0 ? s->xfers[I.xfer_out].dst_rank : -1;
        o.xfer_in = I.xfer_in;
        o.xfer_out = I.xfer_out;
        o.position = I.position;
    }
    return CCL_OK;
}

void ccl_schedule_destroy(ccl_schedule_t s) { delete s; }

ccl_status_t ccl_plan_create(ccl_schedule_t s, int64_t chunk_elems, int32_t dtype, int32_t op,
                             const ccl_plan_opts_t* opts, ccl_plan_t* out)
{
    auto t0 = std::chrono::steady_clock::now();
    if (!s || !out) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    if (op != CCL_SUM) return ccl::fail(CCL_ERR_INVALID_ARG, "only CCL_SUM is supported");
    ccl_plan_opts_t o = merged_opts(opts);
    int ndev = 0;
    CUDA_TRY(cudaGetDeviceCount(&ndev), "cudaGetDeviceCount");
    if (ndev <= 0) return ccl::fail(CCL_ERR_CUDA, "no CUDA device");
    auto* p = new ccl_plan();
    ccl_status_t st = ccl::build_plan(*s, chunk_elems, dtype, o, &p->img);
    if (st != CCL_OK) { delete p; return st; }
    cudaGetDevice(&p->device);
    p->nranks = s->nranks;
    ccl::PlanImage& img = p->img;

    // co-residency: every threadblock of the grid must be resident at once;
    // with the thread count left to the library, halve it until they fit.
    // Shared-memory stages of the bulk path take what the SM has left for
    // the threadblocks it must hold.
    int nsm = 0, per_sm = 0, smem_sm = 0, smem_optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, p->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, p->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device);
    cudaFuncAttributes fa{};
    const void* kfn = ccl::exec_kernel(img.protocol, img.engine);
    if (img.protocol == CCL_PROTO_LL && img.nthreads > ccl::kMaxThreadsLL) {
        if (opts && opts->nthreads) {
            delete p;
            return ccl::fail(CCL_ERR_INVALID_ARG, "plans with the LL protocol use at most 512 threads");
        }
        img.nthreads = ccl::kMaxThreadsLL;
    }
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kfn);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_optin - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) { delete p; return ccl::cuda_fail(e, "device attributes"); }
    const int need_sm = nsm > 0 ? (img.ntb + nsm - 1) / nsm : 1;
    int budget = smem_sm / std::max(1, need_sm) - (int)fa.sharedSizeBytes - 1024;
    budget = std::min(budget, smem_optin - (int)fa.sharedSizeBytes);
    const int64_t stage_bytes = img.tile_bytes;
    // LL plans move every tile through registers
    const bool can_bulk = img.bulk && img.protocol != CCL_PROTO_LL && img.tile_bytes > 0;
    int ns = can_bulk ? (int)std::min<int64_t>(8, budget / stage_bytes) : 0;
    if (ns < 2) ns = 0;
    while (true) {
        size_t dyn = (size_t)ns * stage_bytes;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, img.nthreads, dyn);
        if (e != cudaSuccess) { delete p; return ccl::cuda_fail(e, "occupancy query"); }
        if ((int64_t)per_sm * nsm >= img.ntb) break;
        if (ns > 2) { --ns; continue; }
        if (ns > 0) { ns = 0; continue; }
        if ((opts && opts->nthreads) || img.nthreads <= 128) break;
        img.nthreads = img.nthreads / 2 >= 128 ? img.nthreads / 2 : 128;
        ns = can_bulk ? (int)std::min<int64_t>(8, budget / stage_bytes) : 0;
        if (ns < 2) ns = 0;
    }
    img.ns = ns;
    if ((int64_t)per_sm * nsm < img.ntb) {
        std::string msg = "plan needs " + std::to_string(img.ntb) + " co-resident threadblocks of " +
                          std::to_string(img.nthreads) + " threads; the device holds " + std::to_string(per_sm * nsm);
        delete p;
        return ccl::fail(CCL_ERR_UNSUPPORTED, msg);
    }

    // one blob for the read-only tables
    size_t o_recs = 0;
    size_t o_tb = align_up(o_recs + img.recs.size() * sizeof(ccl::DRec), 256);
    size_t o_links = align_up(o_tb + img.tb_begin.size() * sizeof(int32_t), 256);
    size_t o_deps = align_up(o_links + img.links.size() * sizeof(ccl::DLink), 256);
    size_t blob = align_up(o_deps + std::max<size_t>(1, img.deps.size()) * sizeof(ccl::DDep), 256);
    std::vector<char> h(blob, 0);
    std::memcpy(h.data() + o_recs, img.recs.data(), img.recs.size() * sizeof(ccl::DRec));
    std::memcpy(h.data() + o_tb, img.tb_begin.data(), img.tb_begin.size() * sizeof(int32_t));
    std::memcpy(h.data() + o_links, img.links.data(), img.links.size() * sizeof(ccl::DLink));
    if (!img.deps.empty()) std::memcpy(h.data() + o_deps, img.deps.data(), img.deps.size() * sizeof(ccl::DDep));

#define PLAN_TRY(call, what)                                               \
    do {                                                                   \
        cudaError_t _e = (call);                                           \
        if (_e != cudaSuccess) { free_plan(p); return ccl::cuda_fail(_e, what); } \
    } while (0)

    PLAN_TRY(cudaMalloc(&p->d_blob, blob), "allocate plan tables");
    PLAN_TRY(cudaMemcpy(p->d_blob, h.data(), blob, cudaMemcpyHostToDevice), "upload plan tables");
    p->flags_count = img.links.size() * 2 * img.S + (size_t)img.ncounters;
    PLAN_TRY(cudaMalloc(&p->d_flags, std::max<size_t>(1, p->flags_count) * sizeof(unsigned long long)), "allocate flags");
    PLAN_TRY(cudaMalloc(&p->d_status, 4 * sizeof(int)), "allocate status");
    if (img.fifo_bytes) PLAN_TRY(cudaMalloc(&p->d_fifo, img.fifo_bytes), "allocate link FIFOs");
    if (img.instrument) PLAN_TRY(cudaMalloc(&p->d_timeline, img.steps.size() * 5 * sizeof(unsigned long long)), "allocate timeline");
    int64_t scratch_bytes = img.scratch_elems * img.esize;
    int64_t dev_bytes = blob + p->flags_count * 8 + 16 + img.fifo_bytes;
    for (int r = 0; r < s->nranks; ++r) {
        if (img.scratch_used[r] && scratch_bytes > 0) {
            PLAN_TRY(cudaMalloc(&p->d_scratch[r], scratch_bytes), "allocate scratch");
            dev_bytes += scratch_bytes;
        }
    }
    if (img.instrument) dev_bytes += img.steps.size() * 24;
    p->device_bytes = dev_bytes;
    if (reset_flags(p, 0) != CCL_OK) { free_plan(p); return CCL_ERR_CUDA; }
    PLAN_TRY(cudaDeviceSynchronize(), "plan upload");
#undef PLAN_TRY

    ccl::KParams& k = p->kp;
    k.recs = reinterpret_cast<const ccl::DRec*>(p->d_blob + o_recs);
    k.tb_begin = reinterpret_cast<const int32_t*>(p->d_blob + o_tb);
    k.links = reinterpret_cast<const ccl::DLink*>(p->d_blob + o_links);
    k.deps = reinterpret_cast<const ccl::DDep*>(p->d_blob + o_deps);
    k.flags = p->d_flags;
    k.counters = p->d_flags + img.links.size() * 2 * img.S;
    k.fifo = p->d_fifo;
    k.status = p->d_status;
    k.timeline = p->d_timeline;
    k.m = img.m;
    k.slot_bytes = img.slot_bytes;
    k.ll = img.protocol == CCL_PROTO_LL;
    k.slot_stride = k.ll ? 2 * img.slot_bytes : img.slot_bytes;
    k.tile_bytes = img.tile_bytes;
    k.ns = img.ns;
    k.timeout_ns = (unsigned long long)img.timeout_ms * 1000000ull;
    k.S = img.S;
    for (int r = 0; r < CCL_MAX_RANKS; ++r) k.bufs[2][r] = p->d_scratch[r];
    p->compile_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
    *out = p;
    return CCL_OK;
}

ccl_status_t ccl_execute(ccl_plan_t p, void* const* in_bufs, void* const* out_bufs, void* stream)
{
    if (!p || !in_bufs || !out_bufs) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    const int es = p->img.esize;
    for (int r = 0; r < p->nranks; ++r) {
        if ((p->img.in_elems && !in_bufs[r]) || (p->img.out_elems && !out_bufs[r]))
            return ccl::fail(CCL_ERR_INVALID_ARG, "null buffer for rank " + std::to_string(r));
        if (((uintptr_t)in_bufs[r] | (uintptr_t)out_bufs[r]) % es)
            return ccl::fail(CCL_ERR_INVALID_ARG, "buffer of rank " + std::to_string(r) + " is not element aligned");
        if (p->img.protocol == CCL_PROTO_LL && ((uintptr_t)in_bufs[r] | (uintptr_t)out_bufs[r]) % 16)
            return ccl::fail(CCL_ERR_INVALID_ARG, "the LL protocol needs 16-byte aligned buffers (rank " +
                                                      std::to_string(r) + ")");
    }
    ccl::KParams k = p->kp;
    for (int r = 0; r < p->nranks; ++r) {
        k.bufs[0][r] = static_cast<char*>(in_bufs[r]);
        k.bufs[1][r] = static_cast<char*>(out_bufs[r]);
    }
    // an input that shares memory with an output (in-place AllReduce) is
    // written during the execution: no streaming loads from inputs then
    k.stream_in = 1;
    {
        const size_t ib = (size_t)p->img.in_elems * es, ob = (size_t)p->img.out_elems * es;
        for (int r = 0; r < p->nranks && k.stream_in && ib; ++r)
            for (int q = 0; q < p->nranks && ob; ++q) {
                const char* a = static_cast<const char*>(in_bufs[r]);
                const char* b = static_cast<const char*>(out_bufs[q]);
                if (a < b + ob && b < a + ib) { k.stream_in = 0; break; }
            }
    }
    k.exec = p->exec;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->img.ntb == 0) return CCL_OK;  // empty program: nothing to move
    void* args[] = {&k};
    cudaError_t e = cudaLaunchCooperativeKernel(ccl::exec_kernel(p->img.protocol, p->img.engine), dim3(p->img.ntb),
                                                dim3(p->img.nthreads), args,
                                                (size_t)p->img.ns * p->img.tile_bytes, s);
    if (e != cudaSuccess) return ccl::cuda_fail(e, "executor launch");
    p->exec += 1;
    return CCL_OK;
}

ccl_status_t ccl_execute_host(ccl_plan_t p, const void* const* host_in, void* const* host_out,
                              void* const* dev_in, void* const* dev_out, void* stream)
{
    if (!p || !host_in || !host_out || !dev_in || !dev_out) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t ib = (size_t)p->img.in_elems * p->img.esize, ob = (size_t)p->img.out_elems * p->img.esize;
    for (int r = 0; r < p->nranks; ++r)
        CUDA_TRY(cudaMemcpyAsync(dev_in[r], host_in[r], ib, cudaMemcpyHostToDevice, s), "copy input to device");
    ccl_status_t st = ccl_execute(p, dev_in, dev_out, stream);
    if (st != CCL_OK) return st;
    for (int r = 0; r < p->nranks; ++r)
        CUDA_TRY(cudaMemcpyAsync(host_out[r], dev_out[r], ob, cudaMemcpyDeviceToHost, s), "copy output to host");
    return CCL_OK;
}

ccl_status_t ccl_execute_host_async(ccl_plan_t p, const void* const* host_in, void* const* host_out,
                                    void* const* dev_in, void* const* dev_out, void* copy_in_stream,
                                    void* compute_stream, void* copy_out_stream)
{
    if (!p || !host_in || !host_out || !dev_in || !dev_out) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    cudaStream_t si = static_cast<cudaStream_t>(copy_in_stream);
    cudaStream_t sc = static_cast<cudaStream_t>(compute_stream);
    cudaStream_t so = static_cast<cudaStream_t>(copy_out_stream);
    for (cudaEvent_t* e : {&p->ev_in, &p->ev_k, &p->ev_out})
        if (!*e) CUDA_TRY(cudaEventCreateWithFlags(e, cudaEventDisableTiming), "create pipeline event");
    const size_t ib = (size_t)p->img.in_elems * p->img.esize, ob = (size_t)p->img.out_elems * p->img.esize;
    // the previous call's kernel must be done reading the device inputs
    if (p->pipe_started) CUDA_TRY(cudaStreamWaitEvent(si, p->ev_k, 0), "order input copies");
    for (int r = 0; r < p->nranks; ++r)
        CUDA_TRY(cudaMemcpyAsync(dev_in[r], host_in[r], ib, cudaMemcpyHostToDevice, si), "copy input to device");
    CUDA_TRY(cudaEventRecord(p->ev_in, si), "record input copies");
    CUDA_TRY(cudaStreamWaitEvent(sc, p->ev_in, 0), "order kernel after input copies");
    // and the previous call's output copies done reading the device outputs
    if (p->pipe_started) CUDA_TRY(cudaStreamWaitEvent(sc, p->ev_out, 0), "order kernel after output copies");
    ccl_status_t st = ccl_execute(p, dev_in, dev_out, sc);
    if (st != CCL_OK) return st;
    CUDA_TRY(cudaEventRecord(p->ev_k, sc), "record kernel");
    CUDA_TRY(cudaStreamWaitEvent(so, p->ev_k, 0), "order output copies");
    for (int r = 0; r < p->nranks; ++r)
        CUDA_TRY(cudaMemcpyAsync(host_out[r], dev_out[r], ob, cudaMemcpyDeviceToHost, so), "copy output to host");
    CUDA_TRY(cudaEventRecord(p->ev_out, so), "record output copies");
    p->pipe_started = true;
    return CCL_OK;
}

ccl_status_t ccl_plan_status(ccl_plan_t p)
{
    if (!p) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    int hs[4] = {0, 0, 0, 0};
    CUDA_TRY(cudaMemcpy(hs, p->d_status, sizeof(hs), cudaMemcpyDeviceToHost), "read status");
    if (hs[0] == 0) return CCL_OK;
    static const char* reasons[] = {"?", "dependency counter", "incoming slot", "free outgoing slot",
                                    "its own data warps"};
    std::string msg = "threadblock " + std::to_string(hs[1]) + " (rank " +
                      std::to_string(hs[1] >= 0 && hs[1] < (int)p->img.tb_rank.size() ? p->img.tb_rank[hs[1]] : -1) +
                      ") gave up waiting for " + reasons[(hs[3] >= 1 && hs[3] <= 4) ? hs[3] : 0] + " at step " +
                      std::to_string(hs[2]);
    ccl_status_t code = (ccl_status_t)hs[0];
    if (reset_flags(p, 0) != CCL_OK) return CCL_ERR_CUDA;
    CUDA_TRY(cudaDeviceSynchronize(), "reset after timeout");
    return ccl::fail(code, msg);
}

ccl_status_t ccl_plan_stats(ccl_plan_t p, ccl_plan_stats_t* st)
{
    if (!p || !st) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    fill_stats(p->img, st);
    st->device_bytes = p->device_bytes;
    st->compile_ms = p->compile_ms;
    return CCL_OK;
}

ccl_status_t ccl_plan_check(ccl_schedule_t s, int64_t chunk_elems, int32_t dtype, const ccl_plan_opts_t* opts,
                            ccl_plan_stats_t* st)
{
    auto t0 = std::chrono::steady_clock::now();
    if (!s) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    ccl::PlanImage img;
    ccl_status_t r = ccl::build_plan(*s, chunk_elems, dtype, merged_opts(opts), &img);
    if (r != CCL_OK) return r;
    if (st) {
        fill_stats(img, st);
        st->compile_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
    }
    return CCL_OK;
}

ccl_status_t ccl_schedule_timeline(ccl_schedule_t s, int32_t scheduler, int32_t* xfer_sp, int32_t* nsub)
{
    if (!s) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    if (scheduler != CCL_SCHED_RR && scheduler != CCL_SCHED_HPDS)
        return ccl::fail(CCL_ERR_INVALID_ARG, "unknown scheduler");
    ccl::Timeline tl;
    ccl_status_t r = ccl::build_timeline(*s, scheduler, &tl);
    if (r != CCL_OK) return r;
    if (xfer_sp) std::copy(tl.xfer_sp.begin(), tl.xfer_sp.end(), xfer_sp);
    if (nsub) *nsub = tl.nsp;
    return CCL_OK;
}

ccl_status_t ccl_plan_timeline(ccl_plan_t p, double* idle, int32_t cap, double* mean_idle, double* max_idle,
                               double* span_us)
{
    if (!p) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    if (!p->d_timeline) return ccl::fail(CCL_ERR_INVALID_ARG, "plan was created without instrumentation");
    const ccl::PlanImage& img = p->img;
    if (idle && cap < img.ntb) return ccl::fail(CCL_ERR_INVALID_ARG, "capacity too small");
    CUDA_TRY(cudaDeviceSynchronize(), "synchronize");
    std::vector<unsigned long long> t(img.steps.size() * 5);
    CUDA_TRY(cudaMemcpy(t.data(), p->d_timeline, t.size() * 8, cudaMemcpyDeviceToHost), "read timeline");
    unsigned long long lo = ~0ull, hi = 0;
    for (size_t k = 0; k < img.steps.size(); ++k) {
        lo = std::min(lo, t[5 * k]);
        hi = std::max(hi, t[5 * k + 4]);
    }
    double span = hi > lo ? (double)(hi - lo) : 1.0;
    double sum = 0, mx = 0;
    for (int b = 0; b < img.ntb; ++b) {
        // steps of one threadblock overlap (the issuer runs ahead of the data
        // path): busy time is the length of the union of the intervals from
        // the end of each step's waits to the post of its last tile
        std::vector<std::pair<unsigned long long, unsigned long long>> iv;
        for (int k = img.tb_begin[b]; k < img.tb_begin[b + 1]; ++k) {
            const unsigned long long s0 = t[5 * k] + t[5 * k + 1], s1 = t[5 * k + 4];
            if (s1 > s0) iv.emplace_back(s0, s1);
        }
        std::sort(iv.begin(), iv.end());
        double busy = 0;
        unsigned long long cur0 = 0, cur1 = 0;
        bool open = false;
        for (const auto& e : iv) {
            if (open && e.first <= cur1) {
                cur1 = std::max(cur1, e.second);
                continue;
            }
            if (open) busy += (double)(cur1 - cur0);
            cur0 = e.first;
            cur1 = e.second;
            open = true;
        }
        if (open) busy += (double)(cur1 - cur0);
        double id = std::min(1.0, std::max(0.0, 1.0 - busy / span));
        if (idle) idle[b] = id;
        sum += id;
        mx = std::max(mx, id);
    }
    if (mean_idle) *mean_idle = img.ntb ? sum / img.ntb : 0;
    if (max_idle) *max_idle = mx;
    if (span_us) *span_us = span / 1000.0;
    return CCL_OK;
}

ccl_status_t ccl_plan_timeline_raw(ccl_plan_t p, uint64_t* stamps, int64_t cap, int32_t* tb_begin,
                                   int32_t tb_cap, int64_t* nsteps)
{
    if (!p) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    const ccl::PlanImage& img = p->img;
    if (nsteps) *nsteps = (int64_t)img.steps.size();
    if (tb_begin) {
        if (tb_cap < img.ntb + 1) return ccl::fail(CCL_ERR_INVALID_ARG, "threadblock capacity too small");
        for (int b = 0; b <= img.ntb; ++b) tb_begin[b] = img.tb_begin[b];
    }
    if (!stamps) return CCL_OK;
    if (!p->d_timeline) return ccl::fail(CCL_ERR_INVALID_ARG, "plan was created without instrumentation");
    if (cap < 5 * (int64_t)img.steps.size()) return ccl::fail(CCL_ERR_INVALID_ARG, "capacity too small");
    CUDA_TRY(cudaDeviceSynchronize(), "synchronize");
    CUDA_TRY(cudaMemcpy(stamps, p->d_timeline, img.steps.size() * 5 * 8, cudaMemcpyDeviceToHost), "read timeline");
    return CCL_OK;
}

ccl_status_t ccl_plan_steps(ccl_plan_t p, ccl_step_info_t* out, int64_t cap, int64_t* n)
{
    if (!p) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    const ccl::PlanImage& img = p->img;
    const int64_t ns = (int64_t)img.steps.size();
    if (n) *n = ns;
    if (!out) return CCL_OK;
    if (cap < ns) return ccl::fail(CCL_ERR_INVALID_ARG, "capacity too small");
    const int ch = img.channels > 0 ? img.channels : 1;
    for (int b = 0; b < img.ntb; ++b)
        for (int k = img.tb_begin[b]; k < img.tb_begin[b + 1]; ++k) {
            const ccl::DStep& s = img.steps[k];
            const ccl::DInstr& d = img.instrs[s.instr];
            ccl_step_info_t& o = out[k];
            o.tb = b;
            o.kind = d.kind;
            o.rank = img.tb_rank[b];
            o.channel = s.instr % ch;
            o.mb = s.mb;
            o.link_in = d.link_in;
            o.link_out = d.link_out;
            o.nslots = s.nslots;
            o.dep_count = s.dep_count;
            o.drain = s.drain;
            o.nelem = s.nelem;
        }
    return CCL_OK;
}

ccl_status_t ccl_plan_debug_drop_signal(ccl_plan_t p, int32_t tb, int32_t step)
{
    if (!p) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    ccl::PlanImage& img = p->img;
    if (tb < 0 || tb >= img.ntb) return ccl::fail(CCL_ERR_INVALID_ARG, "threadblock out of range");
    int k = img.tb_begin[tb] + step;
    if (step < 0 || k >= img.tb_begin[tb + 1]) return ccl::fail(CCL_ERR_INVALID_ARG, "step out of range");
    img.steps[k].flags |= ccl::STEP_NOPOST;
    img.recs[k].flags |= ccl::STEP_NOPOST;
    ccl::DRec* dst = const_cast<ccl::DRec*>(p->kp.recs) + k;
    CUDA_TRY(cudaMemcpy(dst, &img.recs[k], sizeof(ccl::DRec), cudaMemcpyHostToDevice), "patch step");
    return CCL_OK;
}

void ccl_plan_destroy(ccl_plan_t p) { free_plan(p); }

}  // extern "C"
