// Ring AllReduce that allocates nothing: its link FIFOs, flags and status
// word live in one file-scope device array instead of plan-owned memory.
//
// This variant has no counterpart in the pages.  It exists for callers that
// must not allocate device memory when they run a collective: code whose
// device memory is entirely pre-reserved by a framework allocator, code
// that cannot afford the device-wide synchronisation a cudaMalloc may cause
// in the middle of a step, and run-after-initialisation code that forbids
// allocation altogether.  Such a caller passes its input and output buffers
// and nothing else.
//
// The threadblock program is the same fused ring program the compiler
// produces for a ring AllReduce (send, recv-reduce-send, recv-reduce-copy-
// send, recv-copy-send, recv), computed in the kernel from (rank, channel,
// step) instead of read from tables, with micro-batch-major order and
// micro-batch pieces of at most half a FIFO.  Reduction order is therefore
// the ring order of the plan path, bit for bit.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "ccl_internal.h"
#include "ccl_core.cuh"

namespace ccl {
namespace {

constexpr int kSlots = 4;                          // FIFO slots per link
constexpr long long kSlotBytes = 32 * 1024;        // bytes per slot
constexpr int kMaxLinks = 64;                      // ranks x channels
constexpr long long kFifoBytes = (long long)kMaxLinks * kSlots * kSlotBytes;   // 8 MiB
constexpr long long kFlagWords = (long long)kMaxLinks * 2 * kSlots;
constexpr long long kStatusBytes = 64;
constexpr long long kScratchBytes = kFifoBytes + kFlagWords * 8 + kStatusBytes;
constexpr unsigned long long kTimeoutNs = 2000000000ull;

// The scratch of every call on this device (8 MiB + 4 KiB, held by every GPU
// that loads the library until the process exits).
static __device__ __align__(256) unsigned char g_ring_scratch[kScratchBytes];

struct StaticParams {
    char* in[CCL_MAX_RANKS];
    char* out[CCL_MAX_RANKS];
    unsigned char* scratch;   // device address of g_ring_scratch
    long long chunk_elems;
    int nranks, channels, dtype;
    int stream_in;            // inputs share no memory with outputs: streaming loads allowed
};

__host__ __device__ inline void piece(long long n, long long ve, long long parts, long long k, long long* off,
                                      long long* len)
{
    long long V = n / ve;
    long long a = (V * k / parts) * ve;
    long long b = (k == parts - 1) ? n : (V * (k + 1) / parts) * ve;
    *off = a;
    *len = b - a;
}

__global__ void __launch_bounds__(512, 2) ring_static_kernel(const __grid_constant__ StaticParams P)
{
    __shared__ int s_abort;
    const int R = P.nranks;
    const int r = blockIdx.x % R;
    const int c = blockIdx.x / R;
    const int es = (P.dtype == CCL_BF16 || P.dtype == CCL_F16) ? 2 : 4;
    const long long ve = 16 / es;
    unsigned long long* flags = reinterpret_cast<unsigned long long*>(P.scratch + kFifoBytes);
    int* status = reinterpret_cast<int*>(P.scratch + kFifoBytes + kFlagWords * 8);
    const int lout = c * R + r;
    const int lin = c * R + (r + R - 1) % R;
    char* fifo_out = reinterpret_cast<char*>(P.scratch) + (long long)lout * kSlots * kSlotBytes;
    const char* fifo_in = reinterpret_cast<const char*>(P.scratch) + (long long)lin * kSlots * kSlotBytes;
    unsigned long long* full_out = flags + (long long)lout * 2 * kSlots;
    unsigned long long* full_in = flags + (long long)lin * 2 * kSlots;
    unsigned long long* free_in = full_in + kSlots;
    unsigned long long* free_out = full_out + kSlots;

    // channel range of a chunk, and micro-batch pieces of at most half a FIFO
    long long coff, clen;
    piece(P.chunk_elems, ve, P.channels, c, &coff, &clen);
    const long long slot_elems = kSlotBytes / es;
    long long cslots = (clen + slot_elems - 1) / slot_elems;
    const long long m = cslots > kSlots / 2 ? (cslots + kSlots / 2 - 1) / (kSlots / 2) : 1;
    unsigned long long seq_in = 0, seq_out = 0, waited = 0;
    const int nsteps = R == 1 ? 1 : 2 * R - 1;
    int si = 0;
    for (long long mb = 0; mb < m; ++mb) {
        long long poff, plen;
        piece(clen, ve, m, mb, &poff, &plen);
        for (int s = 0; s < nsteps; ++s, ++si) {
            // fused ring instruction of this step and the chunk it handles
            int kind, chunk;
            if (R == 1) { kind = CCL_I_COPY; chunk = 0; }
            else if (s == 0) { kind = CCL_I_SEND; chunk = (r + R - 1) % R; }
            else if (s < R - 1) { kind = CCL_I_RRS; chunk = ((r - 1 - s) % R + R) % R; }
            else if (s == R - 1) { kind = CCL_I_RRCS; chunk = r; }
            else if (s < 2 * R - 2) { kind = CCL_I_RCS; chunk = ((r - 1 - (s - R)) % R + R) % R; }
            else { kind = CCL_I_RECV; chunk = (r + 1) % R; }
            const bool rd = kind != CCL_I_SEND && kind != CCL_I_COPY;
            const bool wr = kind == CCL_I_SEND || kind == CCL_I_RRS || kind == CCL_I_RRCS || kind == CCL_I_RCS;
            const bool red = kind == CCL_I_RRS || kind == CCL_I_RRCS;
            const bool has_dst = kind == CCL_I_RRCS || kind == CCL_I_RCS || kind == CCL_I_RECV || kind == CCL_I_COPY;
            const long long base = (long long)chunk * P.chunk_elems + coff + poff;
            const long long nslots = rd || wr ? ((plen + slot_elems - 1) / slot_elems > 0
                                                     ? (plen + slot_elems - 1) / slot_elems : 1)
                                              : 1;
            for (long long k = 0; k < nslots; ++k) {
                const long long e0 = k * slot_elems;
                long long n = plen - e0;
                if (rd || wr) n = n > slot_elems ? slot_elems : n;
                if (n < 0) n = 0;
                const unsigned long long sin = seq_in + k, sout = seq_out + k;
                if (threadIdx.x == 0) {
                    int ok = 1;
                    if (rd) ok = wait_geq(full_in + sin % kSlots, sin + 1, status, kTimeoutNs, si, WAIT_FULL, waited);
                    if (ok && wr && sout + 1 > (unsigned long long)kSlots)
                        ok = wait_geq(free_out + sout % kSlots, sout + 1 - kSlots, status, kTimeoutNs, si,
                                      WAIT_FREE, waited);
                    s_abort = !ok;
                }
                __syncthreads();
                if (s_abort) return;
                const char* slot_in = fifo_in + (long long)(sin % kSlots) * kSlotBytes;
                char* slot_out = fifo_out + (long long)(sout % kSlots) * kSlotBytes;
                const char* a = rd ? slot_in : P.in[r] + (base + e0) * es;
                const char* b = red ? P.in[r] + (base + e0) * es : nullptr;
                char* o1 = has_dst ? P.out[r] + (base + e0) * es : slot_out;
                char* o2 = has_dst && wr ? slot_out : nullptr;
                const bool as = !rd && P.stream_in, bs = P.stream_in;
                if (n > 0) {
                    switch (P.dtype) {
                    case CCL_F32: move_dt<CCL_F32>(red, a, as, b, bs, o1, has_dst, o2, n); break;
                    case CCL_BF16: move_dt<CCL_BF16>(red, a, as, b, bs, o1, has_dst, o2, n); break;
                    case CCL_F16: move_dt<CCL_F16>(red, a, as, b, bs, o1, has_dst, o2, n); break;
                    default: move_dt<CCL_I32>(red, a, as, b, bs, o1, has_dst, o2, n); break;
                    }
                }
                __syncthreads();
                if (threadIdx.x == 0) {
                    if (rd) st_release(free_in + sin % kSlots, sin + 1);
                    if (wr) st_release(full_out + sout % kSlots, sout + 1);
                }
            }
            if (rd) seq_in += nslots;
            if (wr) seq_out += nslots;
        }
    }
}

std::mutex g_mu;
unsigned char* g_addr[64] = {};   // per-device address of g_ring_scratch

}  // namespace
}  // namespace ccl

extern "C" ccl_status_t ccl_allreduce_ring_noalloc(void* const* in_bufs, void* const* out_bufs, int32_t nranks,
                                                   int64_t chunk_elems, int32_t dtype, int32_t channels,
                                                   void* stream)
{
    using namespace ccl;
    if (!in_bufs || !out_bufs) return fail(CCL_ERR_INVALID_ARG, "null buffer array");
    if (nranks < 1 || nranks > CCL_MAX_RANKS) return fail(CCL_ERR_INVALID_ARG, "nranks out of range");
    if (dtype < CCL_F32 || dtype > CCL_I32) return fail(CCL_ERR_INVALID_ARG, "unknown dtype");
    if (chunk_elems <= 0) return fail(CCL_ERR_INVALID_ARG, "chunk_elems must be positive");
    if (channels < 0) return fail(CCL_ERR_INVALID_ARG, "channels must be >= 0");
    if (channels == 0) {
        channels = kMaxLinks / nranks;
        if (channels > 8) channels = 8;
        if (channels < 1) channels = 1;
    }
    if ((long long)nranks * channels > kMaxLinks)
        return fail(CCL_ERR_INVALID_ARG, "nranks * channels = " + std::to_string((long long)nranks * channels) +
                                              " exceeds the " + std::to_string(kMaxLinks) +
                                              " links of the static scratch (" + std::to_string(kScratchBytes) +
                                              " bytes)");
    const int es = (dtype == CCL_BF16 || dtype == CCL_F16) ? 2 : 4;
    for (int r = 0; r < nranks; ++r) {
        if (!in_bufs[r] || !out_bufs[r]) return fail(CCL_ERR_INVALID_ARG, "null buffer for rank " + std::to_string(r));
        if (((uintptr_t)in_bufs[r] | (uintptr_t)out_bufs[r]) % es)
            return fail(CCL_ERR_INVALID_ARG, "buffer of rank " + std::to_string(r) + " is not element aligned");
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(CCL_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(CCL_ERR_UNSUPPORTED, "device index above 63");
    unsigned char* scratch = nullptr;
    {
        // once per device, with that device current: the device address of
        // the array (its host-side name is only a stand-in)
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_addr[dev]) {
            void* ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_ring_scratch);
            if (e != cudaSuccess)
                return fail(CCL_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
            g_addr[dev] = static_cast<unsigned char*>(ptr);
        }
        scratch = g_addr[dev];
    }
    int nsm = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ring_static_kernel, 512, 0);
    if (e != cudaSuccess) return fail(CCL_ERR_CUDA, std::string("occupancy query: ") + cudaGetErrorString(e));
    const int ntb = nranks * channels;
    if ((long long)per_sm * nsm < ntb)
        return fail(CCL_ERR_UNSUPPORTED, "threadblocks cannot be co-resident");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // flags and status restart from zero every call (the FIFO data need not)
    e = cudaMemsetAsync(scratch + kFifoBytes, 0, kFlagWords * 8 + kStatusBytes, s);
    if (e != cudaSuccess) return fail(CCL_ERR_CUDA, std::string("clear flags: ") + cudaGetErrorString(e));
    StaticParams P{};
    for (int r = 0; r < nranks; ++r) {
        P.in[r] = static_cast<char*>(in_bufs[r]);
        P.out[r] = static_cast<char*>(out_bufs[r]);
    }
    // an in-place call (an input shares memory with an output) takes no
    // streaming loads from its inputs
    P.stream_in = 1;
    const size_t bytes = (size_t)nranks * chunk_elems * es;
    for (int r = 0; r < nranks && P.stream_in; ++r)
        for (int q = 0; q < nranks; ++q) {
            const char* a = static_cast<const char*>(in_bufs[r]);
            const char* b = static_cast<const char*>(out_bufs[q]);
            if (a < b + bytes && b < a + bytes) { P.stream_in = 0; break; }
        }
    P.scratch = scratch;
    P.chunk_elems = chunk_elems;
    P.nranks = nranks;
    P.channels = channels;
    P.dtype = dtype;
    void* args[] = {&P};
    e = cudaLaunchCooperativeKernel((const void*)ring_static_kernel, dim3(ntb), dim3(512), args, 0, s);
    if (e != cudaSuccess) return fail(CCL_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(e));
    return CCL_OK;
}
