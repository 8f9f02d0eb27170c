// C ABI entry points, device plan management and the executor kernel.
#include <cuda_runtime.h>
#include <nvrtc.h>

#include <algorithm>
#include <chrono>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "ccl_internal.h"
#include "ccl_plan.h"
#include "ccl_core.cuh"

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

// one instantiation per FIFO protocol and thread limit: only plans with LL
// slots carry the LL data path (no bulk path, at most 512 threads); a
// kernel built for at most 512 threads has twice the registers per thread of
// the 1024-thread one and keeps twice the vectors in flight
constexpr int kMaxThreadsLL = 512;
template <bool LL, int MAXT>
__global__ void __launch_bounds__(MAXT, 1) ccl_exec_kernel(const __grid_constant__ KParams P)
{
    __shared__ __align__(16) CtlShared sh;
    extern __shared__ __align__(128) unsigned char stages[];
    const int b0 = P.tb_begin[blockIdx.x], b1 = P.tb_begin[blockIdx.x + 1];
    ctl_init(P, &sh);
    const int warp = threadIdx.x >> 5;
    if (warp < 3) {
        if ((threadIdx.x & 31) == 0) {
            if (warp == 0) issuer(P, &sh, b0, b1);
            else if (warp == 1) releaser(P, &sh);
            else tma_thread(P, &sh, stages);
        }
        return;
    }
    data_warps<LL, MAXT>(P, &sh);
}

template __global__ void ccl_exec_kernel<false, 1024>(const __grid_constant__ KParams P);
template __global__ void ccl_exec_kernel<false, 512>(const __grid_constant__ KParams P);
template __global__ void ccl_exec_kernel<true, kMaxThreadsLL>(const __grid_constant__ KParams P);

// The library's sequential-engine kernel: thread 0 of every CTA copies the
// step records into shared memory by cp.async, one step ahead (the next
// record travels while the current step runs and has arrived at the barrier
// that ends the step), then the CTA (the cluster) runs each step (seq_step),
// whose leader waits for the step's dependency counters together with its
// first slot.
template <int MAXT>
__global__ void __launch_bounds__(MAXT, 1) ccl_exec_seq_kernel(const __grid_constant__ KParams P)
{
    constexpr int U = InFlight<MAXT>::U;
    __shared__ __align__(16) SeqShared sh;
    const int tid = threadIdx.x;
    const int prog = P.cluster > 1 ? blockIdx.x / P.cluster : blockIdx.x;
    const int b0 = P.tb_begin[prog], b1 = P.tb_begin[prog + 1];
    const unsigned exec_mod = (unsigned)(P.exec % P.S);
    const bool leader = seq_leader(P);
    if (tid == 0 && b0 < b1) {
        prefetch_rec(&sh.rec[0], P.recs + b0);
        asm volatile("cp.async.commit_group;" ::: "memory");
        asm volatile("cp.async.wait_all;" ::: "memory");
    }
    // the program's links, read once (a step's link reads would otherwise
    // go to L2 every step: the acquire fences of the waits drop L1 lines)
    load_prog_links(P, prog, sh.links);
    // every CTA of the cluster has started; the first record and the links
    // are in place
    group_sync(P);
    for (int si = b0; si < b1; ++si) {
        unsigned long long t_start = 0, waited = 0;
        const DRec& st = sh.rec[(si - b0) & 1];
        if (tid == 0 && si + 1 < b1) {
            prefetch_rec(&sh.rec[(si + 1 - b0) & 1], P.recs + si + 1);
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
        if (leader && P.timeline) t_start = gtimer();
        const DLink* Lin = step_link(P, sh.links, st.link_in, st.link_loc & 0xff);
        const DLink* Lout = step_link(P, sh.links, st.link_out, (st.link_loc >> 8) & 0xff);
        seq_step<U>(P, &sh.go, st, Lin, Lout, P.deps + st.dep_begin, st.dep_count, true, si, exec_mod, t_start,
                    waited);
        if (tid == 0) asm volatile("cp.async.wait_all;" ::: "memory");   // the next record is here
        // every thread is done with this record's buffer (it takes the
        // record after next) and sees the next one
        __syncthreads();
    }
}

template __global__ void ccl_exec_seq_kernel<1024>(const __grid_constant__ KParams P);
template __global__ void ccl_exec_seq_kernel<512>(const __grid_constant__ KParams P);

// the executor kernel of an engine and protocol built for at most `build`
// threads (512 or 1024; the LL path has only its 512-thread build)
const void* exec_kernel(int protocol, int engine, int build)
{
    const bool small = build <= 512;
    if (engine == CCL_ENGINE_SEQUENTIAL)
        return small ? (const void*)ccl_exec_seq_kernel<512> : (const void*)ccl_exec_seq_kernel<1024>;
    if (protocol == CCL_PROTO_LL) return (const void*)ccl_exec_kernel<true, kMaxThreadsLL>;
    return small ? (const void*)ccl_exec_kernel<false, 512> : (const void*)ccl_exec_kernel<false, 1024>;
}

}  // namespace ccl

// ======================================================================
// host plan
// ======================================================================
// ======================================================================
// generated kernels: run-time compilation and cache
// ======================================================================
namespace ccl {
extern const char* const kEmbeddedText[];
extern const char* const kEmbeddedName[];
extern const int kEmbeddedCount;
std::string generate_plan_source(const PlanImage& img, int build, std::string* why);

namespace {
std::mutex g_gen_mu;
std::map<std::string, std::vector<char>> g_cubins;   // generated source -> its sm_103a image

// Compile a generated source for sm_103a (the device headers it includes are
// handed over as text); a source compiled before comes from the cache (ms 0)
ccl_status_t compile_generated(const std::string& src, std::vector<char>* cubin, double* ms)
{
    std::lock_guard<std::mutex> lk(g_gen_mu);
    auto it = g_cubins.find(src);
    if (it != g_cubins.end()) {
        *cubin = it->second;
        *ms = 0;
        return CCL_OK;
    }
    const auto t0 = std::chrono::steady_clock::now();
    nvrtcProgram prog;
    if (nvrtcCreateProgram(&prog, src.c_str(), "ccl_gen.cu", kEmbeddedCount, kEmbeddedText, kEmbeddedName) !=
        NVRTC_SUCCESS)
        return fail(CCL_ERR_INTERNAL, "nvrtcCreateProgram failed");
    const char* opts[] = {"--gpu-architecture=sm_103a", "-std=c++17", "-lineinfo"};
    const nvrtcResult r = nvrtcCompileProgram(prog, 3, opts);
    if (r != NVRTC_SUCCESS) {
        size_t n = 0;
        nvrtcGetProgramLogSize(prog, &n);
        std::string log(n, '\0');
        if (n) nvrtcGetProgramLog(prog, &log[0]);
        nvrtcDestroyProgram(&prog);
        if (log.size() > 4000) log.resize(4000);
        return fail(CCL_ERR_INTERNAL, std::string("run-time compilation of the generated kernel failed: ") +
                                          nvrtcGetErrorString(r) + "\n" + log);
    }
    size_t n = 0;
    nvrtcGetCUBINSize(prog, &n);
    cubin->assign(n, 0);
    nvrtcGetCUBIN(prog, cubin->data());
    nvrtcDestroyProgram(&prog);
    g_cubins[src] = *cubin;
    *ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
    return CCL_OK;
}
}  // namespace
}  // namespace ccl

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
    // the plan's own generated kernel (codegen = 1)
    cudaLibrary_t gen_lib = nullptr;
    cudaKernel_t gen_kernel = nullptr;
    double codegen_ms = 0;
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
        o.codegen = opts->codegen;
        o.cluster = opts->cluster;
        o.fold = opts->fold;
    }
    return o;
}

// the kernel a plan launches
const void* launch_fn(const ccl_plan* p)
{
    if (p->gen_kernel) return (const void*)p->gen_kernel;
    return ccl::exec_kernel(p->img.protocol, p->img.engine, p->img.kbuild);
}

// Blocks of `fn` (threads, dynamic shared memory) the device holds at once,
// in units of threadblock programs: CTAs per SM x SMs, or with clusters of
// `cluster` CTAs the clusters that fit.
cudaError_t resident_programs(const void* fn, int threads, size_t dyn, int cluster, int nsm, int ntb, long long* out)
{
    if (cluster <= 1) {
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, dyn);
        *out = (long long)per_sm * nsm;
        return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(ntb * cluster));
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = dyn;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)cluster;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
    *out = n;
    return e;
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
    st->kernel_build = img.kbuild;
    st->cluster = img.cluster;
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
    if (p->gen_lib) cudaLibraryUnload(p->gen_lib);
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
    o->codegen = 0;
    o->cluster = 0;
    o->fold = 3;
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
    if (img.protocol == CCL_PROTO_LL && img.nthreads > ccl::kMaxThreadsLL) {
        if (opts && opts->nthreads) {
            delete p;
            return ccl::fail(CCL_ERR_INVALID_ARG, "plans with the LL protocol use at most 512 threads");
        }
        img.nthreads = ccl::kMaxThreadsLL;
    }
    // both thread-limit builds of the engine take all the shared memory a
    // block may opt in to (the static part of the two is the same)
    for (int nt : {512, 1024}) {
        const void* f = ccl::exec_kernel(img.protocol, img.engine, nt);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, f);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     smem_optin - (int)fa.sharedSizeBytes);
    }
    if (e != cudaSuccess) { delete p; return ccl::cuda_fail(e, "device attributes"); }
    const int need_sm = nsm > 0 ? (img.ntb + nsm - 1) / nsm : 1;
    int budget = smem_sm / std::max(1, need_sm) - (int)fa.sharedSizeBytes - 1024;
    budget = std::min(budget, smem_optin - (int)fa.sharedSizeBytes);
    const int64_t stage_bytes = img.tile_bytes;
    // LL plans move every tile through registers
    const bool can_bulk = img.bulk && img.protocol != CCL_PROTO_LL && img.tile_bytes > 0;
    int ns = can_bulk ? (int)std::min<int64_t>(8, budget / stage_bytes) : 0;
    if (ns < 2) ns = 0;
    // For a thread count of at most 512 the 512-thread build (eight vectors
    // in flight per thread, up to 128 registers) comes first; when its
    // register use leaves too few threadblocks per SM the 1024-thread build
    // (64 registers, four vectors) is tried at the same thread count before
    // stages or threads are given up.
    while (true) {
        size_t dyn = (size_t)ns * stage_bytes;
        bool fit = false;
        for (int build : {512, 1024}) {
            if (build == 512 && img.nthreads > 512) continue;
            long long progs = 0;
            e = resident_programs(ccl::exec_kernel(img.protocol, img.engine, build), img.nthreads, dyn, img.cluster,
                                  nsm, img.ntb, &progs);
            if (e != cudaSuccess) { delete p; return ccl::cuda_fail(e, "occupancy query"); }
            img.kbuild = build;
            per_sm = (int)std::min<long long>(progs / std::max(1, nsm), 1 << 20);
            if (progs >= img.ntb) { fit = true; break; }
        }
        if (fit) break;
        if (ns > 2) { --ns; continue; }
        if (ns > 0) { ns = 0; continue; }
        if ((opts && opts->nthreads) || img.nthreads <= 128) break;
        img.nthreads = img.nthreads / 2 >= 128 ? img.nthreads / 2 : 128;
        ns = can_bulk ? (int)std::min<int64_t>(8, budget / stage_bytes) : 0;
        if (ns < 2) ns = 0;
    }
    img.ns = ns;
    {
        long long progs = 0;
        e = resident_programs(ccl::exec_kernel(img.protocol, img.engine, img.kbuild), img.nthreads,
                              (size_t)ns * stage_bytes, img.cluster, nsm, img.ntb, &progs);
        if (e != cudaSuccess) { delete p; return ccl::cuda_fail(e, "occupancy query"); }
        if (progs < img.ntb) {
            std::string msg = "plan needs " + std::to_string(img.ntb) + " co-resident threadblock programs of " +
                              std::to_string(img.nthreads) + " threads" +
                              (img.cluster > 1 ? " on clusters of " + std::to_string(img.cluster) + " CTAs" : "") +
                              "; the device holds " + std::to_string(progs);
            delete p;
            return ccl::fail(CCL_ERR_UNSUPPORTED, msg);
        }
    }
    if (o.codegen) {
        // the plan's own kernel, built for the same thread limit
        std::string why;
        const std::string src = ccl::generate_plan_source(img, img.kbuild, &why);
        if (src.empty()) {
            delete p;
            return ccl::fail(CCL_ERR_UNSUPPORTED, "no generated kernel for this plan: " + why);
        }
        std::vector<char> cubin;
        st = ccl::compile_generated(src, &cubin, &p->codegen_ms);
        if (st != CCL_OK) { delete p; return st; }
        e = cudaLibraryLoadData(&p->gen_lib, cubin.data(), nullptr, nullptr, 0, nullptr, nullptr, 0);
        if (e == cudaSuccess) e = cudaLibraryGetKernel(&p->gen_kernel, p->gen_lib, "ccl_gen_kernel");
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, (const void*)p->gen_kernel);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute((const void*)p->gen_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     smem_optin - (int)fa.sharedSizeBytes);
        long long gen_progs = 0;
        if (e == cudaSuccess)
            e = resident_programs((const void*)p->gen_kernel, img.nthreads, (size_t)ns * stage_bytes, img.cluster, nsm,
                                  img.ntb, &gen_progs);
        if (e != cudaSuccess) { free_plan(p); return ccl::cuda_fail(e, "load the generated kernel"); }
        if (gen_progs < img.ntb) {
            free_plan(p);
            return ccl::fail(CCL_ERR_UNSUPPORTED, "the generated kernel's threadblocks cannot all be co-resident");
        }
    }

    // one blob for the read-only tables
    size_t o_recs = 0;
    size_t o_tb = align_up(o_recs + img.recs.size() * sizeof(ccl::DRec), 256);
    size_t o_links = align_up(o_tb + img.tb_begin.size() * sizeof(int32_t), 256);
    size_t o_deps = align_up(o_links + img.links.size() * sizeof(ccl::DLink), 256);
    size_t o_plinks = align_up(o_deps + std::max<size_t>(1, img.deps.size()) * sizeof(ccl::DDep), 256);
    size_t blob = align_up(o_plinks + std::max<size_t>(1, img.prog_links.size()) * sizeof(int32_t), 256);
    std::vector<char> h(blob, 0);
    if (!img.prog_links.empty())
        std::memcpy(h.data() + o_plinks, img.prog_links.data(), img.prog_links.size() * sizeof(int32_t));
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
    k.prog_links = reinterpret_cast<const int32_t*>(p->d_blob + o_plinks);
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
    k.cluster = img.cluster;
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
    cudaError_t e;
    if (p->img.cluster > 1) {
        // every program on its own cluster, all of them co-resident
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(p->img.ntb * p->img.cluster));
        cfg.blockDim = dim3((unsigned)p->img.nthreads);
        cfg.dynamicSmemBytes = (size_t)p->img.ns * p->img.tile_bytes;
        cfg.stream = s;
        cudaLaunchAttribute at[2];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = (unsigned)p->img.cluster;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        at[1].id = cudaLaunchAttributeCooperative;
        at[1].val.cooperative = 1;
        cfg.attrs = at;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelExC(&cfg, launch_fn(p), args);
    } else {
        e = cudaLaunchCooperativeKernel(launch_fn(p), dim3(p->img.ntb), dim3(p->img.nthreads), args,
                                        (size_t)p->img.ns * p->img.tile_bytes, s);
    }
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
    st->codegen = p->gen_kernel != nullptr;
    st->codegen_ms = p->codegen_ms;
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

ccl_status_t ccl_plan_codegen_source(ccl_schedule_t s, int64_t chunk_elems, int32_t dtype,
                                     const ccl_plan_opts_t* opts, char* buf, size_t cap, size_t* len,
                                     int32_t compile, int64_t* cubin_bytes)
{
    if (!s) return ccl::fail(CCL_ERR_INVALID_ARG, "null argument");
    ccl::PlanImage img;
    const ccl_plan_opts_t o = merged_opts(opts);
    ccl_status_t r = ccl::build_plan(*s, chunk_elems, dtype, o, &img);
    if (r != CCL_OK) return r;
    std::string why;
    const std::string src = ccl::generate_plan_source(img, img.nthreads <= 512 ? 512 : 1024, &why);
    if (src.empty()) return ccl::fail(CCL_ERR_UNSUPPORTED, "no generated kernel for this plan: " + why);
    if (len) *len = src.size();
    if (buf) {
        if (cap < src.size() + 1) return ccl::fail(CCL_ERR_INVALID_ARG, "capacity too small");
        std::memcpy(buf, src.c_str(), src.size() + 1);
    }
    if (compile) {
        std::vector<char> cubin;
        double ms = 0;
        r = ccl::compile_generated(src, &cubin, &ms);
        if (r != CCL_OK) return r;
        if (cubin_bytes) *cubin_bytes = (int64_t)cubin.size();
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
    if (p->gen_kernel) return ccl::fail(CCL_ERR_UNSUPPORTED, "a generated kernel reads no step records to patch");
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
