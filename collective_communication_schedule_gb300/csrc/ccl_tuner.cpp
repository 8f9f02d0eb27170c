// Tuner: subspace coordinate descent over the resource parameters.
//
// AutoCCL report, "research method" 1-2: implementation parameters (here:
// the threadblock allocation policy -- one per connection, or packed and
// balanced --, the FIFO protocol, the transport and the execution engine --
// pipelined or sequential: sixteen subspaces in all) split the search space
// into small subspaces; inside each, the resource parameters nChannel, nThread and
// chunk size are optimised one coordinate at a time, raising a parameter
// while bandwidth keeps improving (bandwidth is unimodal in each of them).
// Grids: channels {1,2,4,8,12,16,24,32,48}, threads {128,256,512,1024},
// slot size 16 KiB .. 4 MiB in powers of two, on the sequential engine
// CTAs per threadblock program {1,2,4,8}, and with direct transport each
// fold bit {0,1} (receives into senders, copy chains, reduction chains,
// three-hop copy chains).  A probe is the median of
// `reps` CUDA-event-timed executions after one warm-up; a point whose plan
// cannot be built (threadblocks not co-resident, FIFO too small) scores 0.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <map>
#include <tuple>
#include <vector>

#include "ccl_internal.h"

namespace ccl {
namespace {

struct Prober {
    ccl_schedule_t s;
    int64_t ce;
    int32_t dtype;
    void* const* in;
    void* const* out;
    cudaStream_t stream;
    int reps;
    int probes = 0;
    std::map<std::tuple<int, int, int64_t, int, int, int, int, int, int>, double> cache;  // -> microseconds (0 = infeasible)

    double time_us(const ccl_plan_opts_t& o)
    {
        auto key = std::make_tuple(o.channels, o.nthreads, o.slot_bytes, o.tb_alloc, o.protocol, o.link_mode, o.engine,
                                   o.cluster, o.fold);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
        ++probes;
        double us = 0;
        ccl_plan_t p = nullptr;
        if (ccl_plan_create(s, ce, dtype, CCL_SUM, &o, &p) == CCL_OK) {
            cudaEvent_t a, b;
            cudaEventCreate(&a);
            cudaEventCreate(&b);
            std::vector<float> t;
            bool ok = ccl_execute(p, in, out, stream) == CCL_OK;
            for (int k = 0; k < reps && ok; ++k) {
                cudaEventRecord(a, stream);
                ok = ccl_execute(p, in, out, stream) == CCL_OK;
                cudaEventRecord(b, stream);
                cudaEventSynchronize(b);
                float ms = 0;
                cudaEventElapsedTime(&ms, a, b);
                t.push_back(ms);
            }
            cudaStreamSynchronize(stream);
            if (ok && ccl_plan_status(p) == CCL_OK && !t.empty()) {
                std::sort(t.begin(), t.end());
                us = 1000.0 * t[t.size() / 2];
            }
            cudaEventDestroy(a);
            cudaEventDestroy(b);
            ccl_plan_destroy(p);
        }
        cache[key] = us;
        return us;
    }
};

const int kChannels[] = {1, 2, 4, 8, 12, 16, 24, 32, 48};
const int kThreads[] = {128, 256, 512, 1024};

std::vector<int64_t> slot_grid()
{
    std::vector<int64_t> v;
    for (int64_t b = 16 * 1024; b <= 4 * 1024 * 1024; b *= 2) v.push_back(b);
    return v;
}

template <typename T>
int nearest(const std::vector<T>& g, T x)
{
    int best = 0;
    for (int i = 0; i < (int)g.size(); ++i)
        if (std::llabs((long long)g[i] - (long long)x) < std::llabs((long long)g[best] - (long long)x)) best = i;
    return best;
}

}  // namespace
}  // namespace ccl

// Subspace coordinate descent over (channels, threads, slot size) for each
// threadblock-allocation policy; `probe` returns the bandwidth of a point
// (any unit, 0 = infeasible).
extern "C" ccl_status_t ccl_tune_search(const ccl_plan_opts_t* start, const ccl_tune_opts_t* topts,
                                        double (*probe)(void* user, const ccl_plan_opts_t* o), void* user,
                                        ccl_plan_opts_t* best, double* best_bw, int32_t* probes)
{
    using namespace ccl;
    if (!probe || !best) return fail(CCL_ERR_INVALID_ARG, "null argument");
    ccl_tune_opts_t to{3, 5, 0.01, 0};
    if (topts) {
        if (topts->max_rounds > 0) to.max_rounds = topts->max_rounds;
        if (topts->reps > 0) to.reps = topts->reps;
        if (topts->min_gain > 0) to.min_gain = topts->min_gain;
        if (topts->max_channels > 0) to.max_channels = topts->max_channels;
    }
    ccl_plan_opts_t base;
    ccl_plan_opts_default(&base);
    if (start) {
        ccl_plan_opts_t z = *start;
        if (z.channels) base.channels = z.channels;
        if (z.nthreads) base.nthreads = z.nthreads;
        if (z.slot_bytes) base.slot_bytes = z.slot_bytes;
        if (z.fifo_slots) base.fifo_slots = z.fifo_slots;
        base.microbatches = z.microbatches;
        base.scheduler = z.scheduler;
        base.tb_alloc = z.tb_alloc;
        base.mb_order = z.mb_order;
        if (z.tile_bytes) base.tile_bytes = z.tile_bytes;
        if (z.timeout_ms) base.timeout_ms = z.timeout_ms;
        base.bulk = z.bulk;
        base.link_mode = z.link_mode;
        base.channel_scaling = z.channel_scaling;
        base.mb_window = z.mb_window;
        base.protocol = z.protocol;
        base.tb_budget = z.tb_budget;
        base.engine = z.engine;
        base.cluster = z.cluster;
        base.codegen = z.codegen;
        base.fold = z.fold;
    }
    if (!base.nthreads) base.nthreads = 512;
    std::vector<int> gc;
    for (int c : kChannels)
        if (!to.max_channels || c <= to.max_channels) gc.push_back(c);
    if (to.max_channels && (gc.empty() || gc.back() != to.max_channels)) gc.push_back(to.max_channels);
    if (to.max_channels && base.channels > to.max_channels) base.channels = to.max_channels;
    std::vector<int> gt(std::begin(kThreads), std::end(kThreads));
    std::vector<int64_t> gs = slot_grid();
    std::map<std::tuple<int, int, int64_t, int, int, int, int, int, int>, double> cache;
    int nprobe = 0;
    auto measure = [&](const ccl_plan_opts_t& o) {
        auto key = std::make_tuple(o.channels, o.nthreads, o.slot_bytes, o.tb_alloc, o.protocol, o.link_mode, o.engine,
                                   o.cluster, o.fold);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
        ++nprobe;
        double bw = probe(user, &o);
        if (!(bw > 0)) bw = 0;
        cache[key] = bw;
        return bw;
    };
    ccl_plan_opts_t overall = base;
    double overall_bw = measure(base);
    for (int sub = 0; sub < 16; ++sub) {
        ccl_plan_opts_t cur = base;
        // balanced = packed plus merged link-free threadblocks (the same as
        // packed when every threadblock has a FIFO link)
        cur.tb_alloc = sub & 1 ? CCL_TB_BALANCED : CCL_TB_CONNECTION;
        cur.protocol = sub & 2 ? CCL_PROTO_LL : CCL_PROTO_SIMPLE;
        cur.link_mode = sub & 4 ? CCL_LINK_DIRECT : CCL_LINK_FIFO;
        cur.engine = sub & 8 ? CCL_ENGINE_SEQUENTIAL : CCL_ENGINE_PIPELINED;
        // the sequential engine also chooses the CTAs per program (clusters)
        const bool seq = cur.engine == CCL_ENGINE_SEQUENTIAL;
        const std::vector<int> gk = seq ? std::vector<int>{1, 2, 4, 8} : std::vector<int>{1};
        if (!seq) cur.cluster = 0;
        // direct transport also chooses its folds: each of the four fold
        // bits (receives, copy chains, reduction chains, three-hop copy
        // chains) a coordinate of its own with the values 0 and 1
        const bool direct = cur.link_mode == CCL_LINK_DIRECT;
        int ic = nearest(gc, cur.channels), it = nearest(gt, cur.nthreads), is = nearest(gs, cur.slot_bytes);
        int ik = seq ? nearest(gk, std::max(1, cur.cluster)) : 0;
        int fb[4] = {cur.fold & 1, (cur.fold >> 1) & 1, (cur.fold >> 2) & 1, (cur.fold >> 3) & 1};
        auto eval = [&](int c, int t, int sl, int k, const int* f) {
            ccl_plan_opts_t o = cur;
            o.channels = gc[c];
            o.nthreads = gt[t];
            o.slot_bytes = gs[sl];
            o.cluster = gk[k] > 1 ? gk[k] : 0;
            if (direct) o.fold = f[0] | (f[1] << 1) | (f[2] << 2) | (f[3] << 3);
            return measure(o);
        };
        std::vector<int> coords{0, 1, 2};
        if (seq) coords.push_back(3);
        if (direct) for (int b = 0; b < 4; ++b) coords.push_back(4 + b);
        double bw = eval(ic, it, is, ik, fb);
        for (int round = 0; round < to.max_rounds; ++round) {
            bool moved = false;
            for (int coord : coords) {
                int* idx = coord == 0 ? &ic : coord == 1 ? &it : coord == 2 ? &is : coord == 3 ? &ik : &fb[coord - 4];
                int n = coord == 0 ? (int)gc.size() : coord == 1 ? (int)gt.size() : coord == 2 ? (int)gs.size()
                        : coord == 3 ? (int)gk.size() : 2;
                auto at = [&](int v) {
                    if (coord >= 4) {
                        int f[4] = {fb[0], fb[1], fb[2], fb[3]};
                        f[coord - 4] = v;
                        return eval(ic, it, is, ik, f);
                    }
                    return coord == 0 ? eval(v, it, is, ik, fb) : coord == 1 ? eval(ic, v, is, ik, fb)
                           : coord == 2 ? eval(ic, it, v, ik, fb) : eval(ic, it, is, v, fb);
                };
                // raise while bandwidth improves; if the first raise does not
                // help, try lowering the same way
                for (int dir : {+1, -1}) {
                    bool any = false;
                    while (*idx + dir >= 0 && *idx + dir < n) {
                        double nb = at(*idx + dir);
                        if (nb > bw * (1.0 + to.min_gain)) {
                            *idx += dir;
                            bw = nb;
                            any = moved = true;
                        } else {
                            break;
                        }
                    }
                    if (any) break;
                }
            }
            if (!moved) break;
        }
        if (bw > overall_bw) {
            overall_bw = bw;
            overall = cur;
            overall.channels = gc[ic];
            overall.nthreads = gt[it];
            overall.slot_bytes = gs[is];
            overall.cluster = gk[ik] > 1 ? gk[ik] : 0;
            if (direct) overall.fold = fb[0] | (fb[1] << 1) | (fb[2] << 2) | (fb[3] << 3);
        }
    }
    *best = overall;
    if (best_bw) *best_bw = overall_bw;
    if (probes) *probes = nprobe;
    if (!(overall_bw > 0)) return fail(CCL_ERR_UNSUPPORTED, "no configuration could run");
    return CCL_OK;
}

namespace {
double gpu_probe(void* user, const ccl_plan_opts_t* o)
{
    auto* P = static_cast<ccl::Prober*>(user);
    double us = P->time_us(*o);
    return us > 0 ? 1.0 / us : 0.0;
}
}  // namespace

extern "C" ccl_status_t ccl_tune(ccl_schedule_t s, int64_t chunk_elems, int32_t dtype, void* const* in_bufs,
                                 void* const* out_bufs, void* stream, const ccl_tune_opts_t* topts,
                                 const ccl_plan_opts_t* start, ccl_plan_opts_t* best, ccl_tune_report_t* report)
{
    using namespace ccl;
    if (!s || !in_bufs || !out_bufs || !best) return fail(CCL_ERR_INVALID_ARG, "null argument");
    ccl_tune_opts_t to{3, 5, 0.01, 0};
    if (topts) {
        if (topts->max_rounds > 0) to.max_rounds = topts->max_rounds;
        if (topts->reps > 0) to.reps = topts->reps;
        if (topts->min_gain > 0) to.min_gain = topts->min_gain;
        if (topts->max_channels > 0) to.max_channels = topts->max_channels;
    }
    Prober P{s, chunk_elems, dtype, in_bufs, out_bufs, static_cast<cudaStream_t>(stream), to.reps};
    ccl_plan_opts_t base;
    ccl_plan_opts_default(&base);
    if (start) base = *start;
    if (!base.nthreads) base.nthreads = 512;
    if (!base.channels) base.channels = 1;
    if (!base.slot_bytes) base.slot_bytes = 128 * 1024;
    if (!base.fifo_slots) base.fifo_slots = 4;
    if (!base.tile_bytes) base.tile_bytes = 16 * 1024;
    if (!base.timeout_ms) base.timeout_ms = 2000;
    if (to.max_channels && base.channels > to.max_channels) base.channels = to.max_channels;
    double default_us = P.time_us(base);
    double bw = 0;
    int32_t probes = 0;
    ccl_status_t st = ccl_tune_search(&base, &to, gpu_probe, &P, best, &bw, &probes);
    if (report) {
        std::memset(report, 0, sizeof(*report));
        report->probes = P.probes;
        report->best_us = bw > 0 ? 1.0 / bw : 0;
        report->default_us = default_us;
        ccl_plan_t p = nullptr;
        if (st == CCL_OK && ccl_plan_create(s, chunk_elems, dtype, CCL_SUM, best, &p) == CCL_OK) {
            ccl_plan_stats_t ps;
            ccl_plan_stats(p, &ps);
            if (report->best_us > 0) report->best_gbs = ps.schedule_bytes / (report->best_us * 1e3);
            ccl_plan_destroy(p);
        }
    }
    return st;
}

// One tuning per message size (AutoCCL report, research method 1-2: the
// parameters are chosen per message size): rows[i] gets the configuration
// for chunk_elems[i] elements per chunk and its report.  The buffers must
// hold the largest size.
extern "C" ccl_status_t ccl_tune_table(ccl_schedule_t s, int32_t dtype, const int64_t* chunk_elems, int32_t n,
                                       void* const* in_bufs, void* const* out_bufs, void* stream,
                                       const ccl_tune_opts_t* topts, const ccl_plan_opts_t* start,
                                       ccl_tune_row_t* rows)
{
    using namespace ccl;
    if (!s || !chunk_elems || n <= 0 || !rows) return fail(CCL_ERR_INVALID_ARG, "bad arguments");
    for (int i = 0; i < n; ++i) {
        std::memset(&rows[i], 0, sizeof(rows[i]));
        rows[i].chunk_elems = chunk_elems[i];
        ccl_status_t st = ccl_tune(s, chunk_elems[i], dtype, in_bufs, out_bufs, stream, topts, start, &rows[i].best,
                                   &rows[i].report);
        if (st != CCL_OK) return st;
    }
    return CCL_OK;
}
