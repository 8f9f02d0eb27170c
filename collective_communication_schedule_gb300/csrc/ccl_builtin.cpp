// Built-in collective programs, written as chunk programs (copy / reduce on
// chunk ranges, program order) so that they go through the same compiler as
// user programs.
//
//  * Ring AllReduce / AllGather / ReduceScatter (MSCCLang report, §II test
//    cases and §IV.1; AutoCCL report, experiment design: AllGather,
//    ReduceScatter, AllReduce).  Ring direction r -> r+1; chunk c enters the
//    reduce-scatter at rank c+1 and completes at rank c, then circulates in
//    the all-gather starting from rank c.
//  * Hierarchical AllReduce (MSCCLang report, §IV.2; HetCCL summary,
//    methodology 3): intra-group ring reduce-scatter leaving slice i on
//    local rank i, a ring AllReduce of slice i over the groups among ranks
//    g*G+i, and an intra-group ring all-gather.
//  * Two-phase AllToAll (MSCCLang report, §IV.3): blocks for other groups
//    are gathered on the in-group aggregator with the destination's local
//    index, then sent as one batch of G blocks per destination.
//  * AllToNext (MSCCLang report, §II and §IV.4): out[r+1] = in[r]; a pair
//    crossing a group boundary is split into G parts, part j relayed through
//    local rank j on both sides so every link of both groups carries a share.
//  * Uneven AllToAll (per-pair sizes, MoE token exchange): one copy per
//    non-empty (source, destination) pair, in shift order.
#include <algorithm>
#include <string>

#include "ccl_internal.h"

namespace ccl {
namespace {

ccl_op_t mk(int op, int sr, int sb, int so, int dr, int db, int dof, int cnt)
{
    ccl_op_t o;
    o.op = op; o.src_rank = sr; o.src_buf = sb; o.src_off = so;
    o.dst_rank = dr; o.dst_buf = db; o.dst_off = dof; o.count = cnt;
    return o;
}

constexpr int IN = CCL_BUF_IN, OUT = CCL_BUF_OUT, SCR = CCL_BUF_SCRATCH;
constexpr int CP = CCL_OP_COPY, RD = CCL_OP_REDUCE;

int md(int a, int m) { return ((a % m) + m) % m; }

// out := in per chunk, then reduce-scatter and all-gather in place on out
void ring_allreduce(int R, std::vector<ccl_op_t>& v)
{
    for (int r = 0; r < R; ++r)
        for (int c = 0; c < R; ++c) v.push_back(mk(CP, r, IN, c, r, OUT, c, 1));
    for (int step = 0; step + 1 < R; ++step)
        for (int c = 0; c < R; ++c)
            v.push_back(mk(RD, md(c + 1 + step, R), OUT, c, md(c + 2 + step, R), OUT, c, 1));
    for (int step = 0; step + 1 < R; ++step)
        for (int c = 0; c < R; ++c)
            v.push_back(mk(CP, md(c + step, R), OUT, c, md(c + step + 1, R), OUT, c, 1));
}

void ring_allgather(int R, std::vector<ccl_op_t>& v)
{
    for (int r = 0; r < R; ++r) v.push_back(mk(CP, r, IN, 0, r, OUT, r, 1));
    for (int step = 0; step + 1 < R; ++step)
        for (int c = 0; c < R; ++c)
            v.push_back(mk(CP, md(c + step, R), OUT, c, md(c + step + 1, R), OUT, c, 1));
}

// the partial of chunk c rides in scratch chunk c, and lands in out[c]
void ring_reducescatter(int R, std::vector<ccl_op_t>& v)
{
    if (R == 1) { v.push_back(mk(CP, 0, IN, 0, 0, OUT, 0, 1)); return; }
    for (int step = 0; step + 1 < R; ++step) {
        for (int c = 0; c < R; ++c) {
            int from = md(c + 1 + step, R), to = md(c + 2 + step, R);
            int fb = step == 0 ? IN : SCR;
            bool last = step == R - 2;
            int tb = last ? OUT : SCR, toff = last ? 0 : c;
            v.push_back(mk(CP, to, IN, c, to, tb, toff, 1));
            v.push_back(mk(RD, from, fb, c, to, tb, toff, 1));
        }
    }
}

void hier_allreduce(int G, int ng, std::vector<ccl_op_t>& v)
{
    int R = G * ng;
    for (int r = 0; r < R; ++r)
        for (int i = 0; i < G; ++i) v.push_back(mk(CP, r, IN, i * ng, r, OUT, i * ng, ng));
    for (int step = 0; step + 1 < G; ++step)
        for (int g = 0; g < ng; ++g)
            for (int i = 0; i < G; ++i)
                v.push_back(mk(RD, g * G + md(i + 1 + step, G), OUT, i * ng,
                               g * G + md(i + 2 + step, G), OUT, i * ng, ng));
    for (int step = 0; step + 1 < ng; ++step)
        for (int i = 0; i < G; ++i)
            for (int k = 0; k < ng; ++k)
                v.push_back(mk(RD, md(k + 1 + step, ng) * G + i, OUT, i * ng + k,
                               md(k + 2 + step, ng) * G + i, OUT, i * ng + k, 1));
    for (int step = 0; step + 1 < ng; ++step)
        for (int i = 0; i < G; ++i)
            for (int k = 0; k < ng; ++k)
                v.push_back(mk(CP, md(k + step, ng) * G + i, OUT, i * ng + k,
                               md(k + step + 1, ng) * G + i, OUT, i * ng + k, 1));
    for (int step = 0; step + 1 < G; ++step)
        for (int g = 0; g < ng; ++g)
            for (int i = 0; i < G; ++i)
                v.push_back(mk(CP, g * G + md(i + step, G), OUT, i * ng,
                               g * G + md(i + step + 1, G), OUT, i * ng, ng));
}

void alltoall_two_phase(int G, int ng, std::vector<ccl_op_t>& v)
{
    int R = G * ng;
    for (int s = 0; s < R; ++s) {
        int g = s / G;
        for (int d = 0; d < R; ++d) {
            int h = d / G;
            if (h == g) {
                v.push_back(mk(CP, s, IN, d, d, OUT, s, 1));
            } else {
                int agg = g * G + d % G;
                int hp = md(h - g - 1, ng);
                v.push_back(mk(CP, s, IN, d, agg, SCR, hp * G + s % G, 1));
            }
        }
    }
    for (int p = 0; p < R; ++p) {
        int g = p / G, l = p % G;
        for (int h = 0; h < ng; ++h) {
            if (h == g) continue;
            int hp = md(h - g - 1, ng);
            v.push_back(mk(CP, p, SCR, hp * G, h * G + l, OUT, g * G, G));
        }
    }
}

void alltonext(int G, int ng, bool wrap, std::vector<ccl_op_t>& v)
{
    int R = G * ng;
    int pairs = wrap ? R : R - 1;
    for (int r = 0; r < pairs; ++r) {
        int dst = (r + 1) % R;
        int g = r / G, h = dst / G;
        if (g == h) { v.push_back(mk(CP, r, IN, 0, dst, OUT, 0, G)); continue; }
        for (int j = 0; j < G; ++j) {
            int a = g * G + j, b = h * G + j;
            int cr = r, cb = IN;          // current holder of part j
            if (a != r) { v.push_back(mk(CP, cr, cb, j, a, SCR, 0, 1)); cr = a; cb = SCR; }
            int co = cb == IN ? j : 0;
            if (b != dst) {
                v.push_back(mk(CP, cr, cb, co, b, SCR, 1, 1));
                cr = b; cb = SCR; co = 1;
            }
            v.push_back(mk(CP, cr, cb, co, dst, OUT, j, 1));
        }
    }
}

}  // namespace

ccl_status_t alltoallv_program(int R, const int32_t* counts, std::vector<ccl_op_t>* ops, int32_t nchunks[3])
{
    if (R < 1 || R > CCL_MAX_RANKS)
        return fail(CCL_ERR_INVALID_ARG, "nranks must be in 1.." + std::to_string(CCL_MAX_RANKS));
    if (!counts) return fail(CCL_ERR_INVALID_ARG, "null counts");
    // block offsets: rank s's input in destination order, rank d's output
    // in source order
    std::vector<int64_t> in_off((size_t)R * R), out_off((size_t)R * R);
    int64_t max_in = 0, max_out = 0, total = 0;
    for (int s = 0; s < R; ++s) {
        int64_t o = 0;
        for (int d = 0; d < R; ++d) {
            const int32_t c = counts[(size_t)s * R + d];
            if (c < 0) return fail(CCL_ERR_INVALID_ARG, "negative count");
            in_off[(size_t)s * R + d] = o;
            o += c;
        }
        max_in = std::max(max_in, o);
        total += o;
    }
    for (int d = 0; d < R; ++d) {
        int64_t o = 0;
        for (int s = 0; s < R; ++s) {
            out_off[(size_t)s * R + d] = o;
            o += counts[(size_t)s * R + d];
        }
        max_out = std::max(max_out, o);
    }
    if (total == 0) return fail(CCL_ERR_INVALID_ARG, "no chunk to move");
    if (max_in > (1 << 30) || max_out > (1 << 30)) return fail(CCL_ERR_INVALID_ARG, "per-rank total above 2^30 chunks");
    ops->clear();
    for (int k = 0; k < R; ++k)
        for (int s = 0; s < R; ++s) {
            const int d = (s + k) % R;
            const int32_t c = counts[(size_t)s * R + d];
            if (c > 0)
                ops->push_back(mk(CP, s, IN, (int)in_off[(size_t)s * R + d], d, OUT,
                                  (int)out_off[(size_t)s * R + d], c));
        }
    nchunks[0] = (int32_t)max_in;
    nchunks[1] = (int32_t)max_out;
    nchunks[2] = 0;
    return CCL_OK;
}

ccl_status_t builtin_program(int kind, int R, int G, uint32_t flags, std::vector<ccl_op_t>* ops,
                             int32_t nchunks[3])
{
    if (R < 1 || R > CCL_MAX_RANKS)
        return fail(CCL_ERR_INVALID_ARG, "nranks must be in 1.." + std::to_string(CCL_MAX_RANKS));
    ops->clear();
    bool grouped = kind == CCL_HIER_ALLREDUCE || kind == CCL_ALLTOALL_2PHASE || kind == CCL_ALLTONEXT;
    if (grouped && (G < 1 || R % G != 0))
        return fail(CCL_ERR_INVALID_ARG, "group_size must divide nranks");
    int ng = grouped ? R / G : 1;
    switch (kind) {
    case CCL_RING_ALLREDUCE:
        ring_allreduce(R, *ops); nchunks[0] = R; nchunks[1] = R; nchunks[2] = 0; break;
    case CCL_RING_ALLGATHER:
        ring_allgather(R, *ops); nchunks[0] = 1; nchunks[1] = R; nchunks[2] = 0; break;
    case CCL_RING_REDUCESCATTER:
        ring_reducescatter(R, *ops); nchunks[0] = R; nchunks[1] = 1; nchunks[2] = R > 1 ? R : 0;
        break;
    case CCL_HIER_ALLREDUCE:
        hier_allreduce(G, ng, *ops); nchunks[0] = R; nchunks[1] = R; nchunks[2] = 0; break;
    case CCL_ALLTOALL_2PHASE:
        alltoall_two_phase(G, ng, *ops); nchunks[0] = R; nchunks[1] = R;
        nchunks[2] = (ng - 1) * G; break;
    case CCL_ALLTONEXT:
        alltonext(G, ng, (flags & CCL_FLAG_WRAP) != 0, *ops); nchunks[0] = G; nchunks[1] = G;
        nchunks[2] = ng > 1 ? 2 : 0; break;
    default:
        return fail(CCL_ERR_INVALID_ARG, "unknown builtin kind " + std::to_string(kind));
    }
    return CCL_OK;
}

}  // namespace ccl
