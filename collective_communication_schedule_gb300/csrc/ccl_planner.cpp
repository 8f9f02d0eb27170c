// Planner: compiled schedule + execution parameters -> threadblock programs.
//
// Steps (ReSCCL report, §II.1-II.2; MSCCLang report, §III.1):
//  1. Task timeline.  A task is one cross-rank transfer (it occupies the link
//     between its two ranks) or one rank-local instruction.  A task waits for
//     the tasks of every instruction its sender or receiver depends on, and
//     a transfer that is forwarded waits for the transfer it forwards.  Tasks
//     are list-scheduled into sub-pipelines; one sub-pipeline never holds two
//     tasks on the same link and never a task with a predecessor in the same
//     sub-pipeline.  RR takes ready tasks in program order; HPDS
//     (hierarchical-priority dynamic scheduling) takes first the tasks of the
//     chunk that has been scheduled least often.
//  2. Threadblock allocation.  CONNECTION: first fit, one threadblock holds at
//     most one incoming and one outgoing link (one threadblock per
//     connection).  PACKED (state-based): connection threadblocks of a rank
//     whose sets of active sub-pipelines are disjoint are merged.
//  3. Program order inside a threadblock: by sub-pipeline, then program
//     position.  The program is cut into segments, each run micro-batch-major
//     (for every micro-batch, every instruction of the segment) -- the
//     pipelining of MSCCLang's runtime -- and the segments one after the
//     other, which is ReSCCL's task-level execution.  ALGO cuts only where the
//     epoch changes (a whole-instruction dependency lies between), SEGMENT also
//     at idle gaps of the threadblock's timeline, TASK before every
//     instruction.  Inside a segment the micro-batches may be taken in
//     windows of w: every instruction of the segment in turn runs the w
//     micro-batches of the window, so a threadblock holds w independent
//     pieces of one instruction while the piece its next instruction needs
//     is still upstream (w = 1: strictly micro-batch-major).
//  4. Geometry.  Every instruction range is split into `channels` pieces and
//     every channel piece into `m` micro-batch pieces, both in 16-byte units
//     (the element tail goes to the last piece); a piece moves through the
//     link FIFO in slots of `slot_bytes`.
//  5. A link FIFO joins one sending threadblock to one receiving threadblock
//     (one per connection and channel).  Sequence numbers follow the sender's
//     order; a receiver waits for the number of the piece it needs, so the
//     flags are per slot and no piece is read out of turn.
//  6. Dependencies between instructions in different threadblocks become
//     counter waits (per micro-batch when the ranges are identical, on the
//     whole instruction otherwise).
//  7. The programs are executed abstractly with bounded FIFOs; a plan that
//     cannot finish is rejected.
#include <algorithm>
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <set>
#include <string>

#include "ccl_plan.h"

namespace ccl {
namespace {

struct Piece {
    int64_t off, len;
};

Piece split(int64_t n, int64_t ve, int64_t parts, int64_t k)
{
    int64_t V = n / ve;
    int64_t a = (V * k / parts) * ve;
    int64_t b = (k == parts - 1) ? n : (V * (k + 1) / parts) * ve;
    return {a, b - a};
}

int esize_of(int dt) { return (dt == CCL_BF16 || dt == CCL_F16) ? 2 : 4; }

}  // namespace

namespace {

int log_level()
{
    const char* v = std::getenv("CCL_LOG_LEVEL");
    return v ? std::atoi(v) : 0;
}

// One pass of the list scheduler.  split = false: a task waits for every
// task of each instruction its instructions depend on.  split = true: it
// waits only for the task that carries the buffer effects of that
// instruction -- its receive when it has one (a fused receive-...-send
// reads and writes its buffers when the data arrives; its send only passes
// that data on), else its send, else the local task -- so a dependent of a
// fused receive need not wait for the forwarded transfer, whose receiver
// may itself wait for the dependent.
ccl_status_t timeline_pass(const ccl_schedule& s, int scheduler, bool split, Timeline* tl)
{
    const int ni = (int)s.instrs.size();
    const int nx = (int)s.xfers.size();
    // tasks: transfers first, then local instructions
    std::vector<std::vector<int>> itasks(ni);
    struct T {
        int key, a, b, chunk;
        std::vector<int> preds;
        int sp = -1;
    };
    std::vector<T> tasks;
    for (int x = 0; x < nx; ++x) {
        const Xfer& X = s.xfers[x];
        tasks.push_back(T{X.op_index, X.src_rank, X.dst_rank, X.chunk_id, {}});
        itasks[X.send_instr].push_back(x);
        itasks[X.recv_instr].push_back(x);
    }
    // local task of every instruction without a transfer, and in the split
    // model also of a copy-send: its local copy is its buffer effect
    std::vector<int> local_task(ni, -1);
    for (int i = 0; i < ni; ++i) {
        const Instr& I = s.instrs[i];
        const bool copy_part = split && I.xfer_in < 0 && I.xfer_out >= 0 && I.dst.valid();
        if (!itasks[i].empty() && !copy_part) continue;
        local_task[i] = (int)tasks.size();
        itasks[i].push_back(local_task[i]);
        tasks.push_back(T{I.position, -1, -1, (int)I.src.off, {}});
    }
    std::vector<std::vector<int>> ideps(ni);
    for (const Dep& d : s.deps) ideps[d.to].push_back(d.from);
    auto effect_task = [&](int j) {
        const Instr& J = s.instrs[j];
        if (J.xfer_in >= 0) return J.xfer_in;
        return local_task[j] >= 0 ? local_task[j] : J.xfer_out;
    };
    auto add_preds_of = [&](int t, int instr) {
        for (int j : ideps[instr]) {
            if (split) {
                const int u = effect_task(j);
                if (u != t) tasks[t].preds.push_back(u);
                continue;
            }
            for (int u : itasks[j])
                if (u != t) tasks[t].preds.push_back(u);
        }
    };
    for (int x = 0; x < nx; ++x) {
        const Xfer& X = s.xfers[x];
        add_preds_of(x, X.send_instr);
        add_preds_of(x, X.recv_instr);
        int y = s.instrs[X.send_instr].xfer_in;
        if (y >= 0) tasks[x].preds.push_back(y);
        // the send of a copy-send passes on what its local copy reads
        if (local_task[X.send_instr] >= 0) tasks[x].preds.push_back(local_task[X.send_instr]);
    }
    for (int i = 0; i < ni; ++i)
        if (local_task[i] >= 0) add_preds_of(local_task[i], i);
    for (auto& t : tasks) {
        std::sort(t.preds.begin(), t.preds.end());
        t.preds.erase(std::unique(t.preds.begin(), t.preds.end()), t.preds.end());
    }
    const int nt = (int)tasks.size();
    std::vector<int> order(nt);
    for (int i = 0; i < nt; ++i) order[i] = i;
    std::sort(order.begin(), order.end(),
              [&](int a, int b) { return tasks[a].key != tasks[b].key ? tasks[a].key < tasks[b].key : a < b; });
    std::map<int, int> times;  // chunk -> tasks already scheduled
    int done = 0, sp = 0;
    while (done < nt) {
        std::vector<int> ready;
        for (int t : order) {
            if (tasks[t].sp >= 0) continue;
            bool ok = true;
            for (int u : tasks[t].preds)
                if (tasks[u].sp < 0 || tasks[u].sp >= sp) { ok = false; break; }
            if (ok) ready.push_back(t);
        }
        if (ready.empty()) {
            if (split && log_level() >= 2) {
                // the tasks left and the predecessors they still wait for
                for (int t = 0; t < nt; ++t) {
                    if (tasks[t].sp >= 0) continue;
                    std::fprintf(stderr, "[ccl] task %d (%s %d>%d, instructions", t, t < nx ? "transfer" : "local",
                                 tasks[t].a, tasks[t].b);
                    for (int i = 0; i < ni; ++i)
                        for (int u : itasks[i])
                            if (u == t)
                                std::fprintf(stderr, " %d:k%d:r%d:p%d", i, s.instrs[i].kind, s.instrs[i].rank,
                                             s.instrs[i].position);
                    std::fprintf(stderr, ") waits for");
                    for (int u : tasks[t].preds)
                        if (tasks[u].sp < 0) std::fprintf(stderr, " %d", u);
                    std::fprintf(stderr, "\n");
                }
            }
            return fail(CCL_ERR_CYCLE, "dependency cycle among compiled instructions");
        }
        if (scheduler == CCL_SCHED_HPDS) {
            std::stable_sort(ready.begin(), ready.end(), [&](int a, int b) {
                int ca = times[tasks[a].chunk], cb = times[tasks[b].chunk];
                if (ca != cb) return ca < cb;
                if (tasks[a].chunk != tasks[b].chunk) return tasks[a].chunk < tasks[b].chunk;
                return false;
            });
        }
        std::set<std::pair<int, int>> used;
        std::vector<int> chosen;
        for (int t : ready) {
            if (tasks[t].a >= 0) {
                auto key = std::make_pair(tasks[t].a, tasks[t].b);
                if (used.count(key)) continue;
                used.insert(key);
            }
            chosen.push_back(t);
        }
        for (int t : chosen) {
            tasks[t].sp = sp;
            times[tasks[t].chunk]++;
        }
        done += (int)chosen.size();
        ++sp;
    }
    tl->nsp = sp;
    tl->xfer_sp.assign(nx, -1);
    for (int x = 0; x < nx; ++x) tl->xfer_sp[x] = tasks[x].sp;
    tl->sp_lo.assign(ni, 1 << 30);
    tl->sp_hi.assign(ni, -1);
    tl->sp_key.assign(ni, 0);
    for (int i = 0; i < ni; ++i) {
        for (int t : itasks[i]) {
            tl->sp_lo[i] = std::min(tl->sp_lo[i], tasks[t].sp);
            tl->sp_hi[i] = std::max(tl->sp_hi[i], tasks[t].sp);
        }
        // program order inside a threadblock: a dependent's tasks all come
        // after the tasks it waits for, so this key never puts a consumer
        // before its producer
        tl->sp_key[i] = split ? tasks[effect_task(i)].sp : tl->sp_hi[i];
    }
    tl->split = split;
    return CCL_OK;
}

}  // namespace

ccl_status_t build_timeline(const ccl_schedule& s, int scheduler, Timeline* tl)
{
    // whole instructions as the unit first; the finer model only when the
    // coarse one sees a cycle through a fused receive-...-send
    ccl_status_t st = timeline_pass(s, scheduler, false, tl);
    if (st != CCL_ERR_CYCLE) return st;
    return timeline_pass(s, scheduler, true, tl);
}

namespace {

// rank-level threadblocks: list of instruction ids in program order
using TBList = std::vector<std::vector<int>>;

void allocate_connection(const ccl_schedule& s, const Timeline& tl, TBList* tbs, std::vector<int>* tb_rank)
{
    const int ni = (int)s.instrs.size();
    std::vector<std::vector<int>> byrank(s.nranks);
    for (int i = 0; i < ni; ++i) byrank[s.instrs[i].rank].push_back(i);
    for (int r = 0; r < s.nranks; ++r) {
        auto& v = byrank[r];
        std::sort(v.begin(), v.end(), [&](int a, int b) {
            if (tl.sp_key[a] != tl.sp_key[b]) return tl.sp_key[a] < tl.sp_key[b];
            return s.instrs[a].position < s.instrs[b].position;
        });
        struct C { int in, out, id; };
        std::vector<C> cs;
        for (int i : v) {
            const Instr& I = s.instrs[i];
            int in = I.xfer_in >= 0 ? s.xfers[I.xfer_in].src_rank : -1;
            int out = I.xfer_out >= 0 ? s.xfers[I.xfer_out].dst_rank : -1;
            // a copy into another rank's buffer (direct transport) is a
            // connection of its own to that rank
            if ((I.kind == CCL_I_COPY || I.kind == CCL_I_REDUCE || I.kind == CCL_I_REDUCE2) && I.dst.valid() &&
                I.dst.rank != I.rank)
                out = CCL_MAX_RANKS + I.dst.rank;
            // (a two-destination copy: its first remote destination)
            if (I.kind == CCL_I_COPY2) {
                if (I.dst.valid() && I.dst.rank != I.rank) out = CCL_MAX_RANKS + I.dst.rank;
                else if (I.loc.valid() && I.loc.rank != I.rank) out = CCL_MAX_RANKS + I.loc.rank;
            }
            // a folded recv-reduce-copy-send writes the next rank directly
            // but keeps its incoming link: it joins the threadblock of that
            // link (no outgoing connection of its own)
            auto compat = [&](const C& c) {
                return (in < 0 || c.in < 0 || c.in == in) && (out < 0 || c.out < 0 || c.out == out);
            };
            int pick = -1;
            for (int k = 0; k < (int)cs.size() && pick < 0; ++k)
                if (compat(cs[k]) && ((in >= 0 && cs[k].in == in) || (out >= 0 && cs[k].out == out)))
                    pick = k;
            for (int k = 0; k < (int)cs.size() && pick < 0; ++k)
                if (compat(cs[k])) pick = k;
            if (pick < 0) {
                cs.push_back(C{-1, -1, (int)tbs->size()});
                tbs->push_back({});
                tb_rank->push_back(r);
                pick = (int)cs.size() - 1;
            }
            if (in >= 0) cs[pick].in = in;
            if (out >= 0) cs[pick].out = out;
            (*tbs)[cs[pick].id].push_back(i);
        }
    }
}

void pack_state_based(const ccl_schedule& s, const Timeline& tl, TBList* tbs, std::vector<int>* tb_rank)
{
    struct G { int rank; std::vector<char> busy; std::vector<int> instrs; int first; };
    std::vector<int> idx(tbs->size());
    for (size_t i = 0; i < idx.size(); ++i) idx[i] = (int)i;
    auto first_sp = [&](int t) {
        int f = 1 << 30;
        for (int i : (*tbs)[t]) f = std::min(f, tl.sp_lo[i]);
        return f;
    };
    std::sort(idx.begin(), idx.end(), [&](int a, int b) {
        int fa = first_sp(a), fb = first_sp(b);
        return fa != fb ? fa < fb : a < b;
    });
    std::vector<G> groups;
    for (int t : idx) {
        std::vector<char> busy(tl.nsp + 1, 0);
        for (int i : (*tbs)[t])
            for (int k = tl.sp_lo[i]; k <= tl.sp_hi[i]; ++k) busy[k] = 1;
        int pick = -1;
        for (int g = 0; g < (int)groups.size() && pick < 0; ++g) {
            if (groups[g].rank != (*tb_rank)[t]) continue;
            bool clash = false;
            for (int k = 0; k <= tl.nsp && !clash; ++k) clash = busy[k] && groups[g].busy[k];
            if (!clash) pick = g;
        }
        if (pick < 0) {
            groups.push_back(G{(*tb_rank)[t], busy, (*tbs)[t], first_sp(t)});
        } else {
            for (int k = 0; k <= tl.nsp; ++k) groups[pick].busy[k] |= busy[k];
            auto& v = groups[pick].instrs;
            v.insert(v.end(), (*tbs)[t].begin(), (*tbs)[t].end());
        }
    }
    // keep threadblocks grouped by rank
    std::stable_sort(groups.begin(), groups.end(), [](const G& a, const G& b) { return a.rank < b.rank; });
    tbs->clear();
    tb_rank->clear();
    for (auto& g : groups) {
        std::sort(g.instrs.begin(), g.instrs.end(), [&](int a, int b) {
            if (tl.sp_key[a] != tl.sp_key[b]) return tl.sp_key[a] < tl.sp_key[b];
            return s.instrs[a].position < s.instrs[b].position;
        });
        tbs->push_back(g.instrs);
        tb_rank->push_back(g.rank);
    }
}

// Balanced allocation: the instructions of threadblocks that run only
// link-free instructions (local copies, direct copies: no FIFO, so any number
// of them may share a threadblock, and one threadblock's may be split) are
// spread over at most `cap` threadblocks, largest first into the least
// loaded (bytes in chunk units).  A link-free instruction needs no particular
// rank's threadblock, so the bins take instructions of every rank; inside a
// bin instructions run longest dependent chain first, then by sub-pipeline
// and program position.  Binning instructions rather than whole
// threadblocks matters when there are a few more threadblocks than bins
// (21 connections of 8 parts over 19 bins: two bins would carry 16 parts,
// the rest about 9).  The rank of a merged threadblock is that of its
// largest part (reporting only).
void balance_linkfree(const ccl_schedule& s, const Timeline& tl, TBList* tbs, std::vector<int>* tb_rank, int cap)
{
    struct B { int rank; std::vector<int> instrs; int64_t load; int64_t top; };
    std::vector<B> out;
    std::vector<int> free_tbs;
    for (size_t t = 0; t < tbs->size(); ++t) {
        bool link_free = true;
        for (int i : (*tbs)[t]) link_free = link_free && s.instrs[i].xfer_in < 0 && s.instrs[i].xfer_out < 0;
        if (link_free) free_tbs.push_back((int)t);
        else out.push_back(B{(*tb_rank)[t], (*tbs)[t], 0, 0});
    }
    if ((int)free_tbs.size() <= cap) {
        for (int t : free_tbs) out.push_back(B{(*tb_rank)[t], (*tbs)[t], 0, 0});
    } else {
        std::vector<std::pair<int, int>> items;   // (instruction, rank)
        for (int t : free_tbs)
            for (int i : (*tbs)[t]) items.push_back({i, (*tb_rank)[t]});
        std::stable_sort(items.begin(), items.end(), [&](const std::pair<int, int>& a, const std::pair<int, int>& b) {
            return s.instrs[a.first].count > s.instrs[b.first].count;
        });
        std::vector<B> bins(cap, B{-1, {}, 0, 0});
        for (const auto& it : items) {
            int k = 0;
            for (int b = 1; b < cap; ++b)
                if (bins[b].load < bins[k].load) k = b;
            const int64_t w = s.instrs[it.first].count;
            bins[k].instrs.push_back(it.first);
            bins[k].load += w;
            if (w > bins[k].top) {
                bins[k].top = w;
                bins[k].rank = it.second;
            }
        }
        // inside a bin, the instructions with the longest chain of
        // dependent instructions after them first (a relay's first hop
        // before a large independent copy: the copy would hold the chain
        // back); a producer's chain is longer than its consumer's, so the
        // order respects dependencies in and across bins
        const int ni = (int)s.instrs.size();
        std::vector<std::vector<int>> pred(ni);
        std::vector<int> nsucc(ni, 0);
        auto edge = [&](int a, int b) {
            pred[b].push_back(a);
            ++nsucc[a];
        };
        for (const Dep& e : s.deps) edge(e.from, e.to);
        for (const Xfer& X : s.xfers)
            if (X.send_instr >= 0 && X.recv_instr >= 0) edge(X.send_instr, X.recv_instr);
        // from the sinks back (the graph is acyclic: the timeline was built)
        std::vector<int> height(ni, 0), todo;
        for (int i = 0; i < ni; ++i)
            if (nsucc[i] == 0) todo.push_back(i);
        while (!todo.empty()) {
            const int j = todo.back();
            todo.pop_back();
            for (int i : pred[j]) {
                height[i] = std::max(height[i], height[j] + 1);
                if (--nsucc[i] == 0) todo.push_back(i);
            }
        }
        for (auto& b : bins) {
            std::sort(b.instrs.begin(), b.instrs.end(), [&](int a, int c) {
                if (height[a] != height[c]) return height[a] > height[c];
                if (tl.sp_key[a] != tl.sp_key[c]) return tl.sp_key[a] < tl.sp_key[c];
                if (s.instrs[a].position != s.instrs[c].position)
                    return s.instrs[a].position < s.instrs[c].position;
                return a < c;
            });
            out.push_back(std::move(b));
        }
    }
    std::stable_sort(out.begin(), out.end(), [](const B& a, const B& b) { return a.rank < b.rank; });
    tbs->clear();
    tb_rank->clear();
    for (auto& b : out) {
        tbs->push_back(std::move(b.instrs));
        tb_rank->push_back(b.rank);
    }
}

// Epoch of every instruction: the largest number of whole-instruction
// dependencies (partly overlapping ranges) on a path into it, following
// same-rank dependencies and transfers.  Such a dependency needs every
// micro-batch of its producer, so a micro-batch-major segment never spans two
// epochs; because the epoch is a property of the instruction, both ends of a
// link agree on where their segments break.
std::vector<int> epochs(const ccl_schedule& s)
{
    const int ni = (int)s.instrs.size();
    std::vector<std::vector<std::pair<int, int>>> out(ni);   // (to, weight)
    std::vector<int> indeg(ni, 0), ep(ni, 0);
    for (const Dep& d : s.deps) { out[d.from].push_back({d.to, d.exact ? 0 : 1}); ++indeg[d.to]; }
    for (const Xfer& x : s.xfers) { out[x.send_instr].push_back({x.recv_instr, 0}); ++indeg[x.recv_instr]; }
    std::vector<int> q;
    for (int i = 0; i < ni; ++i)
        if (!indeg[i]) q.push_back(i);
    for (size_t h = 0; h < q.size(); ++h) {
        int i = q[h];
        for (auto& e : out[i]) {
            ep[e.first] = std::max(ep[e.first], ep[i] + e.second);
            if (--indeg[e.first] == 0) q.push_back(e.first);
        }
    }
    return ep;
}

// segments of one threadblock program
std::vector<std::vector<int>> make_segments(const Timeline& tl, const std::vector<int>& prog, int order,
                                            const std::vector<int>& ep)
{
    std::vector<std::vector<int>> segs;
    int cur_hi = -1, cur_ep = -1;
    for (int i : prog) {
        bool cut = segs.empty() || ep[i] != cur_ep || order == CCL_MB_TASK ||
                   (order == CCL_MB_SEGMENT && tl.sp_lo[i] > cur_hi + 1);
        if (cut) {
            segs.push_back({});
            cur_hi = -1;
            cur_ep = ep[i];
        }
        segs.back().push_back(i);
        cur_hi = std::max(cur_hi, tl.sp_hi[i]);
    }
    return segs;
}

void fill_records(PlanImage* img)
{
    img->recs.assign(img->steps.size(), DRec{});
    for (size_t k = 0; k < img->steps.size(); ++k) {
        const DStep& st = img->steps[k];
        const DInstr& in = img->instrs[st.instr];
        DRec& r = img->recs[k];
        r.kind = in.kind; r.dtype = in.dtype; r.link_in = in.link_in; r.link_out = in.link_out;
        r.src_buf = in.src_buf; r.src_rank = in.src_rank;
        r.loc_buf = in.loc_buf; r.loc_rank = in.loc_rank;
        r.dst_buf = in.dst_buf; r.dst_rank = in.dst_rank;
        r.nslots = st.nslots; r.dep_begin = st.dep_begin; r.dep_count = st.dep_count;
        r.signal = st.signal; r.mb = st.mb; r.flags = st.flags; r.drain = st.drain;
        r.src_off = in.src_off + st.elem_off;
        r.loc_off = in.loc_off + st.elem_off;
        r.dst_off = in.dst_off + st.elem_off;
        r.x_buf = in.x_buf; r.x_rank = in.x_rank;
        r.x_off = in.x_buf >= 0 ? in.x_off + st.elem_off : 0;
        r.nelem = st.nelem; r.seq_in = st.seq_in; r.seq_out = st.seq_out;
        r.seq_in_mod = (int32_t)(st.seq_in % img->S);
        r.seq_out_mod = (int32_t)(st.seq_out % img->S);
    }
    // every program's first kSeqLinks distinct links, in order of first use,
    // and each step's entries in that table
    img->prog_links.assign((size_t)img->ntb * kSeqLinks, -1);
    for (int b = 0; b < img->ntb; ++b) {
        int32_t* tab = &img->prog_links[(size_t)b * kSeqLinks];
        int n = 0;
        auto entry = [&](int link) {
            if (link < 0) return 0;
            for (int i = 0; i < n; ++i)
                if (tab[i] == link) return i + 1;
            if (n == kSeqLinks) return 0;
            tab[n] = link;
            return ++n;
        };
        for (int k = img->tb_begin[b]; k < img->tb_begin[b + 1]; ++k) {
            DRec& r = img->recs[k];
            r.link_loc = entry(r.link_in) | (entry(r.link_out) << 8);
        }
    }
}

// Parallelization factor of every instruction: `p` for all, or (scaled)
// proportional to the instruction's size, at least 1, so that small
// instructions do not claim as many threadblocks as large ones.  Both ends
// of a transfer have the same size and therefore the same factor.
std::vector<int> channel_counts(const ccl_schedule& s, int p, int scaled)
{
    std::vector<int> pc(s.instrs.size(), p);
    if (!scaled) return pc;
    int64_t cmax = 1;
    for (const Instr& I : s.instrs) cmax = std::max<int64_t>(cmax, I.count);
    for (size_t i = 0; i < s.instrs.size(); ++i) {
        int64_t v = (p * s.instrs[i].count + cmax / 2) / cmax;
        pc[i] = (int)std::max<int64_t>(1, std::min<int64_t>(p, v));
    }
    return pc;
}

struct Attempt {
    int alloc, m, order;
};

ccl_status_t build_image(const ccl_schedule& s, const Timeline& tl, const TBList& tbs,
                         const std::vector<int>& tb_rank, int64_t ce, int dtype,
                         const ccl_plan_opts_t& o, int m, int order, int window, PlanImage* img)
{
    const int ni = (int)s.instrs.size();
    const int p = o.channels;
    const int es = esize_of(dtype);
    const int64_t ve = 16 / es;
    const int S = o.fifo_slots;
    const int64_t slot_elems = o.slot_bytes / es;
    const int nT = (int)tbs.size();

    const std::vector<int> ep = epochs(s);
    const std::vector<int> pc = channel_counts(s, p, o.channel_scaling);

    img->instrs.assign((size_t)ni * p, DInstr{});
    img->steps.clear();
    img->links.clear();
    img->deps.clear();
    img->tb_begin.clear();
    img->tb_rank.clear();
    img->tb_segs.clear();
    img->m = m;
    img->channels = p;
    img->mb_order = order;
    img->mb_window = window;
    img->protocol = o.protocol;
    img->S = S;
    // an LL slot carries slot_bytes of data in twice as many bytes of lines
    const int64_t slot_stride = o.protocol == CCL_PROTO_LL ? 2 * o.slot_bytes : o.slot_bytes;
    img->slot_bytes = o.slot_bytes;
    img->tile_bytes = o.tile_bytes;
    img->bulk = o.engine == CCL_ENGINE_SEQUENTIAL ? 0 : o.bulk;
    img->engine = o.engine;
    img->link_mode = o.link_mode;
    img->nthreads = o.nthreads;
    img->dtype = dtype;
    img->esize = es;
    img->chunk_elems = ce;
    img->nsubpipelines = tl.nsp;
    img->timeout_ms = o.timeout_ms;
    img->instrument = o.instrument;
    for (int r = 0; r < CCL_MAX_RANKS; ++r) img->scratch_used[r] = false;

    // threadblock of every channel instruction: channel ch of rank-level
    // threadblock t is a device threadblock when some instruction of t has
    // that channel; device threadblocks are numbered channel-major
    std::vector<int> tb_of_tc((size_t)nT * p, -1), tb_t, tb_ch;
    for (int ch = 0; ch < p; ++ch)
        for (int t = 0; t < nT; ++t) {
            bool any = false;
            for (int i : tbs[t]) any = any || pc[i] > ch;
            if (!any) continue;
            tb_of_tc[(size_t)t * p + ch] = (int)tb_t.size();
            tb_t.push_back(t);
            tb_ch.push_back(ch);
        }
    const int ntb = (int)tb_t.size();
    std::vector<int> dev_tb_of((size_t)ni * p, -1);
    for (int t = 0; t < nT; ++t)
        for (int i : tbs[t])
            for (int ch = 0; ch < pc[i]; ++ch) dev_tb_of[(size_t)i * p + ch] = tb_of_tc[(size_t)t * p + ch];

    // one FIFO per (sending threadblock, receiving threadblock): every link
    // has a single producer and a single consumer
    std::map<std::pair<int, int>, int> link_id;
    auto get_link = [&](int a, int b, int ch, int stb, int rtb) {
        auto key = std::make_pair(stb, rtb);
        auto it = link_id.find(key);
        if (it != link_id.end()) return it->second;
        int id = (int)img->links.size();
        DLink L{};
        L.slot_base = (int64_t)id * S * slot_stride;
        L.total = 0;
        L.flag_base = id * 2 * S;
        L.src_rank = a; L.dst_rank = b; L.total_mod = 0;
        img->links.push_back(L);
        link_id[key] = id;
        return id;
    };

    // channel instructions
    int64_t sched_bytes = 0;
    for (int i = 0; i < ni; ++i) {
        const Instr& I = s.instrs[i];
        int64_t n = I.count * ce;
        for (int ch = 0; ch < pc[i]; ++ch) {
            Piece pce = split(n, ve, pc[i], ch);
            DInstr& D = img->instrs[(size_t)i * p + ch];
            D.kind = I.kind;
            D.dtype = dtype;
            if (I.xfer_in >= 0) {
                const Xfer& X = s.xfers[I.xfer_in];
                D.link_in = get_link(X.src_rank, I.rank, ch, dev_tb_of[(size_t)X.send_instr * p + ch],
                                     dev_tb_of[(size_t)i * p + ch]);
            } else {
                D.link_in = -1;
            }
            if (I.xfer_out >= 0) {
                const Xfer& X = s.xfers[I.xfer_out];
                D.link_out = get_link(I.rank, X.dst_rank, ch, dev_tb_of[(size_t)i * p + ch],
                                      dev_tb_of[(size_t)X.recv_instr * p + ch]);
            } else {
                D.link_out = -1;
            }
            D.src_rank = I.src.rank; D.src_buf = I.src.valid() ? I.src.buf : -1;
            D.loc_rank = I.loc.rank; D.loc_buf = I.loc.valid() ? I.loc.buf : -1;
            D.dst_rank = I.dst.rank; D.dst_buf = I.dst.valid() ? I.dst.buf : -1;
            D.src_off = I.src.valid() ? I.src.off * ce + pce.off : 0;
            D.loc_off = I.loc.valid() ? I.loc.off * ce + pce.off : 0;
            D.dst_off = I.dst.valid() ? I.dst.off * ce + pce.off : 0;
            D.x_rank = I.x.rank; D.x_buf = I.x.valid() ? I.x.buf : -1;
            D.x_off = I.x.valid() ? I.x.off * ce + pce.off : 0;
            D.nelem = pce.len;
            sched_bytes += kind_bytes_factor(I.kind) * pce.len * es;
            for (const Range* rg : {&I.src, &I.loc, &I.dst, &I.x})
                if (rg->valid() && rg->buf == CCL_BUF_SCRATCH) img->scratch_used[rg->rank] = true;
        }
    }
    img->schedule_bytes = sched_bytes;

    // Inputs that some instruction writes (a program may write into an
    // input buffer): their reads must see data other threadblocks wrote
    // during the execution, so they take no streaming (L1-allocating) load
    // and a bulk copy from them is ordered after generic-proxy writes; inputs
    // nobody writes are read once and streamed.
    std::vector<char> in_written(s.nranks, 0);
    for (const Instr& I : s.instrs) {
        if (I.dst.valid() && I.dst.buf == CCL_BUF_IN) in_written[I.dst.rank] = 1;
        if (I.kind == CCL_I_COPY2 && I.loc.valid() && I.loc.buf == CCL_BUF_IN) in_written[I.loc.rank] = 1;
        if (I.kind == CCL_I_RRC2 && I.src.valid() && I.src.buf == CCL_BUF_IN) in_written[I.src.rank] = 1;
        if (I.x.valid() && I.x.buf == CCL_BUF_IN) in_written[I.x.rank] = 1;
    }
    auto stream_bits = [&](const DInstr& D) {
        int32_t f = 0;
        if (D.kind != CCL_I_RRC2 && D.src_buf == CCL_BUF_IN && !in_written[D.src_rank]) f |= STEP_SRC_STREAM;
        if (D.kind != CCL_I_COPY2 && D.loc_buf == CCL_BUF_IN && !in_written[D.loc_rank]) f |= STEP_LOC_STREAM;
        return f;
    };

    // threadblock programs -> steps
    img->ntb = ntb;
    std::vector<std::vector<int>> step_of((size_t)ni * p, std::vector<int>(m, -1));
    for (int dtb = 0; dtb < ntb; ++dtb) {
        {
            const int t = tb_t[dtb], ch = tb_ch[dtb];
            img->tb_begin.push_back((int)img->steps.size());
            img->tb_rank.push_back(tb_rank[t]);
            std::vector<int> prog;
            for (int i : tbs[t])
                if (pc[i] > ch) prog.push_back(i);
            auto segs = make_segments(tl, prog, order, ep);
            img->tb_segs.emplace_back();
            for (auto& seg : segs) {
                SegInfo sg;
                for (int i : seg) sg.cis.push_back(i * p + ch);
                sg.window = window;
                img->tb_segs.back().push_back(std::move(sg));
            }
            // window by window; inside a window instruction-major
            for (auto& seg : segs) {
                for (int w0 = 0; w0 < m; w0 += window) {
                    const int w1 = std::min(m, w0 + window);
                    for (int i : seg) for (int mb = w0; mb < w1; ++mb) {
                        int ci = i * p + ch;
                        const DInstr& D = img->instrs[ci];
                        Piece pc = split(D.nelem, ve, m, mb);
                        DStep st{};
                        st.instr = ci;
                        st.mb = mb;
                        st.elem_off = pc.off;
                        st.nelem = pc.len;
                        st.seq_in = st.seq_out = 0;
                        bool linked = D.link_in >= 0 || D.link_out >= 0;
                        st.nslots = linked ? (int32_t)std::max<int64_t>(1, (pc.len + slot_elems - 1) / slot_elems) : 0;
                        st.dep_begin = 0;
                        st.dep_count = 0;
                        st.signal = -1;
                        st.flags = stream_bits(D);
                        st.drain = -1;
                        step_of[ci][mb] = (int)img->steps.size();
                        img->steps.push_back(st);
                    }
                }
            }
        }
    }
    img->tb_begin.push_back((int)img->steps.size());

    // sequence numbers per link, in the sending threadblock's order
    {
        std::vector<std::vector<std::pair<int, int>>> senders(img->links.size());  // (step, tb)
        for (int tb = 0; tb < ntb; ++tb)
            for (int k = img->tb_begin[tb]; k < img->tb_begin[tb + 1]; ++k) {
                const DInstr& D = img->instrs[img->steps[k].instr];
                if (D.link_out >= 0) senders[D.link_out].push_back({k, tb});
            }
        for (size_t L = 0; L < senders.size(); ++L) {
            auto& v = senders[L];
            bool single = true;
            for (auto& e : v) single = single && e.second == v[0].second;
            if (!single) {
                std::stable_sort(v.begin(), v.end(), [&](const std::pair<int, int>& a, const std::pair<int, int>& b) {
                    int ia = a.first - img->tb_begin[a.second], ib = b.first - img->tb_begin[b.second];
                    return ia != ib ? ia < ib : a.second < b.second;
                });
            }
            int64_t seq = 0;
            for (auto& e : v) {
                DStep& st = img->steps[e.first];
                st.seq_out = seq;
                seq += st.nslots;
            }
            img->links[L].total = seq;
            img->links[L].total_mod = (int32_t)(seq % S);
        }
        // receivers take the sender's numbers
        for (int i = 0; i < ni; ++i) {
            const Instr& I = s.instrs[i];
            if (I.xfer_in < 0) continue;
            int snd = s.xfers[I.xfer_in].send_instr;
            for (int ch = 0; ch < pc[i]; ++ch)
                for (int mb = 0; mb < m; ++mb) {
                    DStep& r = img->steps[step_of[(size_t)i * p + ch][mb]];
                    const DStep& w = img->steps[step_of[(size_t)snd * p + ch][mb]];
                    if (r.nslots != w.nslots || r.nelem != w.nelem)
                        return fail(CCL_ERR_INTERNAL, "sender and receiver pieces disagree");
                    r.seq_in = w.seq_out;
                }
        }
    }

    // dependencies across threadblocks -> counters
    {
        std::vector<int> counter_of((size_t)ni * p, -1);
        auto counter = [&](int ci) {
            if (counter_of[ci] < 0) counter_of[ci] = img->ncounters++;
            return counter_of[ci];
        };
        img->ncounters = 0;
        std::vector<std::vector<DDep>> waits(img->steps.size());
        for (const Dep& d : s.deps) {
            for (int ch = 0; ch < pc[d.to]; ++ch) {
                int cb = d.to * p + ch;
                // a producer in the same threadblock comes earlier in its
                // program; its tiles must have left the data path before the
                // consumer starts: the same micro-batch of the same channel
                // when the ranges are identical, every piece otherwise
                const bool same_range = d.exact && pc[d.from] == pc[d.to];
                for (int ch2 = 0; ch2 < pc[d.from]; ++ch2) {
                    const int ca2 = d.from * p + ch2;
                    if (dev_tb_of[ca2] != dev_tb_of[cb] || (same_range && ch2 != ch)) continue;
                    int all = -1;
                    for (int mb = 0; mb < m; ++mb) all = std::max(all, step_of[ca2][mb]);
                    for (int mb = 0; mb < m; ++mb) {
                        DStep& c = img->steps[step_of[cb][mb]];
                        const int need = same_range ? step_of[ca2][mb] : all;
                        if (need >= step_of[cb][mb])
                            return fail(CCL_ERR_DEADLOCK, "a producer follows its consumer in one threadblock");
                        c.drain = std::max(c.drain, need);
                    }
                }
                if (d.exact && pc[d.from] == pc[d.to]) {
                    int ca = d.from * p + ch;
                    if (dev_tb_of[ca] == dev_tb_of[cb]) continue;
                    for (int mb = 0; mb < m; ++mb)
                        waits[step_of[cb][mb]].push_back(DDep{counter(ca), 0, mb + 1});
                } else {
                    // all micro-batches of every channel of `from`; the first
                    // step of `to` (micro-batch 0) waits, later ones follow it
                    for (int ch2 = 0; ch2 < pc[d.from]; ++ch2) {
                        int ca = d.from * p + ch2;
                        if (dev_tb_of[ca] == dev_tb_of[cb]) continue;
                        waits[step_of[cb][0]].push_back(DDep{counter(ca), 0, (int64_t)m});
                    }
                }
            }
        }
        for (size_t k = 0; k < img->steps.size(); ++k) {
            auto& w = waits[k];
            std::sort(w.begin(), w.end(), [](const DDep& a, const DDep& b) {
                return a.counter != b.counter ? a.counter < b.counter : a.value > b.value;
            });
            std::vector<DDep> u;
            for (auto& e : w)
                if (u.empty() || u.back().counter != e.counter) u.push_back(e);
            img->steps[k].dep_begin = (int32_t)img->deps.size();
            img->steps[k].dep_count = (int32_t)u.size();
            img->deps.insert(img->deps.end(), u.begin(), u.end());
        }
        for (size_t k = 0; k < img->steps.size(); ++k) {
            int ci = img->steps[k].instr;
            img->steps[k].signal = counter_of[ci];
        }
    }
    img->fifo_bytes = (int64_t)img->links.size() * S * slot_stride;
    fill_records(img);
    return CCL_OK;
}

}  // namespace

bool simulate_plan(const PlanImage& img, std::string* why)
{
    const int ntb = img.ntb;
    const int S = img.S;
    std::vector<int64_t> flags((size_t)img.links.size() * 2 * S, 0);
    std::vector<int64_t> counters(img.ncounters, 0);
    std::vector<int> si(ntb), slot(ntb, 0);
    std::vector<char> deps_ok(ntb, 0);
    for (int t = 0; t < ntb; ++t) si[t] = img.tb_begin[t];
    int finished = 0;
    for (int t = 0; t < ntb; ++t)
        if (si[t] == img.tb_begin[t + 1]) ++finished;
    while (finished < ntb) {
        bool progress = false;
        for (int t = 0; t < ntb; ++t) {
            while (si[t] < img.tb_begin[t + 1]) {
                const DStep& st = img.steps[si[t]];
                const DInstr& D = img.instrs[st.instr];
                if (!deps_ok[t]) {
                    bool ok = true;
                    for (int k = 0; k < st.dep_count && ok; ++k) {
                        const DDep& d = img.deps[st.dep_begin + k];
                        ok = counters[d.counter] >= d.value;
                    }
                    if (!ok) break;
                    deps_ok[t] = 1;
                }
                bool blocked = false;
                while (slot[t] < st.nslots) {
                    int64_t sin = st.seq_in + slot[t], sout = st.seq_out + slot[t];
                    if (D.link_in >= 0) {
                        const DLink& L = img.links[D.link_in];
                        if (flags[L.flag_base + sin % S] < sin + 1) { blocked = true; break; }
                    }
                    if (D.link_out >= 0) {
                        const DLink& L = img.links[D.link_out];
                        if (flags[L.flag_base + S + sout % S] < sout - S + 1) { blocked = true; break; }
                    }
                    if (D.link_in >= 0) {
                        const DLink& L = img.links[D.link_in];
                        flags[L.flag_base + S + sin % S] = sin + 1;
                    }
                    if (D.link_out >= 0) {
                        const DLink& L = img.links[D.link_out];
                        flags[L.flag_base + sout % S] = sout + 1;
                    }
                    ++slot[t];
                    progress = true;
                }
                if (blocked) break;
                if (st.signal >= 0) counters[st.signal] = std::max<int64_t>(counters[st.signal], st.mb + 1);
                ++si[t];
                slot[t] = 0;
                deps_ok[t] = 0;
                progress = true;
                if (si[t] == img.tb_begin[t + 1]) ++finished;
            }
        }
        if (!progress) {
            if (std::getenv("CCL_LOG_LEVEL") && std::atoi(std::getenv("CCL_LOG_LEVEL")) >= 2) {
                for (int t = 0; t < ntb; ++t) {
                    if (si[t] == img.tb_begin[t + 1]) continue;
                    const DStep& st = img.steps[si[t]];
                    const DInstr& D = img.instrs[st.instr];
                    std::fprintf(stderr, "[ccl] stuck tb %d step %d instr %d kind %d mb %d slot %d/%d deps_ok %d",
                                 t, si[t] - img.tb_begin[t], st.instr, D.kind, st.mb, slot[t], st.nslots, deps_ok[t]);
                    if (!deps_ok[t])
                        for (int k = 0; k < st.dep_count; ++k) {
                            const DDep& d = img.deps[st.dep_begin + k];
                            if (counters[d.counter] < d.value)
                                std::fprintf(stderr, " dep(c%d>=%lld have %lld)", d.counter, (long long)d.value,
                                             (long long)counters[d.counter]);
                        }
                    if (D.link_in >= 0)
                        std::fprintf(stderr, " in(L%d seq %lld full %lld)", D.link_in, (long long)(st.seq_in + slot[t]),
                                     (long long)flags[img.links[D.link_in].flag_base + (st.seq_in + slot[t]) % S]);
                    if (D.link_out >= 0)
                        std::fprintf(stderr, " out(L%d seq %lld consumed %lld)", D.link_out,
                                     (long long)(st.seq_out + slot[t]),
                                     (long long)flags[img.links[D.link_out].flag_base + S + (st.seq_out + slot[t]) % S]);
                    std::fprintf(stderr, "\n");
                }
            }
            if (why) {
                for (int t = 0; t < ntb; ++t) {
                    if (si[t] == img.tb_begin[t + 1]) continue;
                    const DStep& st = img.steps[si[t]];
                    const DInstr& D = img.instrs[st.instr];
                    *why = "threadblock " + std::to_string(t) + " (rank " + std::to_string(img.tb_rank[t]) +
                           ") stuck at step " + std::to_string(si[t] - img.tb_begin[t]) + " kind " +
                           std::to_string(D.kind) + " micro-batch " + std::to_string(st.mb) + " slot " +
                           std::to_string(slot[t]) + " of " + std::to_string(st.nslots);
                    break;
                }
            }
            return false;
        }
    }
    return true;
}

namespace {

void dump_programs(const ccl_schedule& s, const Timeline& tl, const TBList& tbs, const std::vector<int>& tr, int m,
                   int order)
{
    static const char* kn[] = {"copy", "reduce", "send", "recv", "rrc", "rcs", "fwd", "rrs", "rrcs", "copy_send"};
    std::fprintf(stderr, "[ccl] m=%d order=%d threadblocks=%zu sub-pipelines=%d\n", m, order, tbs.size(), tl.nsp);
    for (size_t t = 0; t < tbs.size(); ++t) {
        std::fprintf(stderr, "[ccl] tb %zu rank %d:", t, tr[t]);
        for (int i : tbs[t]) {
            const Instr& I = s.instrs[i];
            int pin = I.xfer_in >= 0 ? s.xfers[I.xfer_in].src_rank : -1;
            int pout = I.xfer_out >= 0 ? s.xfers[I.xfer_out].dst_rank : -1;
            std::fprintf(stderr, " %s(i%d %d>%d sp%d-%d)", kn[I.kind], i, pin, pout, tl.sp_lo[i], tl.sp_hi[i]);
        }
        std::fprintf(stderr, "\n");
    }
}

}  // namespace

// Direct transport: a plain send from a buffer whose transfer ends in a plain
// receive into a buffer becomes one copy run by the sender's threadblock
// straight into the receiver's destination; the receive disappears and
// every dependency on it moves to the copy.  Nothing is staged in a FIFO.
ccl_schedule direct_transport(const ccl_schedule& s, int* ndirect, bool fold)
{
    ccl_schedule d = s;
    const int ni = (int)s.instrs.size();
    std::vector<int> redirect(ni);
    for (int i = 0; i < ni; ++i) redirect[i] = i;
    std::vector<char> drop_x(s.xfers.size(), 0), drop_i(ni, 0);
    int n = 0;
    for (size_t x = 0; x < s.xfers.size(); ++x) {
        const Xfer& X = s.xfers[x];
        const Instr& snd = s.instrs[X.send_instr];
        const Instr& rcv = s.instrs[X.recv_instr];
        const bool foldable = snd.kind == CCL_I_COPY_SEND || snd.kind == CCL_I_RRCS || snd.kind == CCL_I_RRCS3 ||
                              snd.kind == CCL_I_RCSEND;
        if ((snd.kind != CCL_I_SEND && !(fold && foldable)) || rcv.kind != CCL_I_RECV) continue;
        Instr& c = d.instrs[X.send_instr];
        if (snd.kind == CCL_I_SEND) {
            c.kind = CCL_I_COPY;
            c.dst = rcv.dst;
        } else if (snd.kind == CCL_I_COPY_SEND) {
            // the copy-send writes its own destination and, in the same
            // pass, the receiver's (held in the local-operand range)
            c.kind = CCL_I_COPY2;
            c.loc = rcv.dst;
        } else if (snd.kind == CCL_I_RRCS) {
            // the recv-reduce-copy-send likewise (its source range, unused:
            // the first operand is the incoming slot)
            c.kind = CCL_I_RRC2;
            c.src = rcv.dst;
        } else {
            // a folded reduction step that sends its result on writes the
            // receiver's destination as its second destination instead
            c.kind = snd.kind == CCL_I_RRCS3 ? CCL_I_RRC3D : CCL_I_REDUCE2;
            c.x = rcv.dst;
        }
        c.xfer_out = -1;
        drop_x[x] = 1;
        drop_i[X.recv_instr] = 1;
        redirect[X.recv_instr] = X.send_instr;
        ++n;
    }
    *ndirect = n;
    if (!n) return d;
    // renumber instructions and transfers
    std::vector<int> inew(ni, -1), xnew(s.xfers.size(), -1);
    std::vector<Instr> instrs;
    for (int i = 0; i < ni; ++i)
        if (!drop_i[i]) { inew[i] = (int)instrs.size(); instrs.push_back(d.instrs[i]); }
    std::vector<Xfer> xfers;
    for (size_t x = 0; x < s.xfers.size(); ++x)
        if (!drop_x[x]) { xnew[x] = (int)xfers.size(); xfers.push_back(s.xfers[x]); }
    for (auto& I : instrs) {
        if (I.xfer_in >= 0) I.xfer_in = xnew[I.xfer_in];
        if (I.xfer_out >= 0) I.xfer_out = xnew[I.xfer_out];
    }
    for (auto& X : xfers) {
        X.send_instr = inew[X.send_instr];
        X.recv_instr = inew[X.recv_instr];
    }
    std::set<std::tuple<int, int, int>> seen;
    std::vector<Dep> deps;
    for (const Dep& e : s.deps) {
        int a = inew[redirect[e.from]], b = inew[redirect[e.to]];
        if (a < 0 || b < 0 || a == b) continue;
        if (!seen.insert(std::make_tuple(a, b, e.exact ? 1 : 0)).second) continue;
        deps.push_back(Dep{a, b, e.exact});
    }
    d.instrs = std::move(instrs);
    d.xfers = std::move(xfers);
    d.deps = std::move(deps);
    return d;
}

// Copy chains (after direct transport): a direct copy c2 that sends on,
// unchanged, exactly the range another direct copy c1 wrote into c2's rank
// is run by c1's pass instead -- one read written to both destinations (a
// CCL_I_COPY2 holding the second destination in its local-operand range)
// instead of c1's write and c2's read-back and write; with depth 3 the copy
// that forwards the second destination joins as well (a CCL_I_COPY3, its
// third destination in the x range).  A ring AllGather's k copy hops become
// ceil(k/2) (ceil(k/3)) steps.  c1 takes over c2's dependencies in
// both directions; c2's writes then happen at c1's time, which is sound
// when every instruction c2 waited for can come before c1 -- a pair whose
// merged dependencies would close a cycle is left alone.  Pairs are formed
// in dependency order (smallest index first among the ready ones), so each
// chain pairs up from its head.
int fold_copy_chains(ccl_schedule& d, int depth)
{
    const int ni = (int)d.instrs.size();
    std::vector<std::set<int>> succ(ni), pred(ni);
    std::map<std::pair<int, int>, int> exact;   // bit 0: an exact edge, bit 1: a non-exact one
    auto add_edge = [&](int a, int b, bool ex) {
        if (a == b) return;
        succ[a].insert(b);
        pred[b].insert(a);
        exact[{a, b}] |= ex ? 1 : 2;
    };
    for (const Dep& e : d.deps) add_edge(e.from, e.to, e.exact);
    for (const Xfer& X : d.xfers)
        if (X.send_instr >= 0 && X.recv_instr >= 0) {
            succ[X.send_instr].insert(X.recv_instr);
            pred[X.recv_instr].insert(X.send_instr);
        }
    // topological order, smallest index first
    std::vector<int> indeg(ni), order;
    std::set<int> ready;
    for (int i = 0; i < ni; ++i)
        if ((indeg[i] = (int)pred[i].size()) == 0) ready.insert(i);
    while (!ready.empty()) {
        const int i = *ready.begin();
        ready.erase(ready.begin());
        order.push_back(i);
        for (int j : succ[i])
            if (--indeg[j] == 0) ready.insert(j);
    }
    if ((int)order.size() != ni) return 0;   // cyclic already: the timeline reports it
    auto direct_copy = [&](int i) {
        const Instr& I = d.instrs[i];
        return I.kind == CCL_I_COPY && I.xfer_in < 0 && I.xfer_out < 0 && I.src.valid() && I.dst.valid() &&
               I.dst.rank != I.rank;
    };
    std::vector<char> gone(ni, 0);
    std::vector<int> mark(ni, -1);
    int nfold = 0, epoch = 0;
    for (int c1 : order) {
        if (gone[c1] || !direct_copy(c1)) continue;
        // up to `depth` destinations: each fold takes the copy that forwards
        // the step's last destination
        for (int held = 1; held < depth; ++held) {
            const Instr& A = d.instrs[c1];
            const Range last = held == 1 ? A.dst : A.loc;
            bool folded = false;
            for (int c2 : std::vector<int>(succ[c1].begin(), succ[c1].end())) {
                if (gone[c2] || !direct_copy(c2)) continue;
                const Instr& B = d.instrs[c2];
                if (!B.src.same(last) || B.count != A.count || B.dst.overlaps(A.src) || B.dst.overlaps(A.dst) ||
                    (held == 2 && B.dst.overlaps(A.loc)))
                    continue;
                // every other instruction c2 waits for must not follow c1
                std::vector<int> stack{c1};
                bool cycle = false;
                mark[c1] = ++epoch;
                while (!stack.empty() && !cycle) {
                    const int v = stack.back();
                    stack.pop_back();
                    for (int w : succ[v]) {
                        if (w == c2 || mark[w] == epoch) continue;
                        if (pred[c2].count(w)) { cycle = true; break; }
                        mark[w] = epoch;
                        stack.push_back(w);
                    }
                }
                if (cycle) continue;
                Instr& F = d.instrs[c1];
                if (held == 1) {
                    F.kind = CCL_I_COPY2;
                    F.loc = B.dst;
                } else {
                    F.kind = CCL_I_COPY3;
                    F.x = B.dst;
                }
                for (int x : std::vector<int>(pred[c2].begin(), pred[c2].end())) {
                    const int ex = exact[{x, c2}];
                    succ[x].erase(c2);
                    if (x == c1) continue;
                    if (ex & 1) add_edge(x, c1, true);
                    if (ex & 2) add_edge(x, c1, false);
                }
                for (int y : std::vector<int>(succ[c2].begin(), succ[c2].end())) {
                    const int ex = exact[{c2, y}];
                    pred[y].erase(c2);
                    if (ex & 1) add_edge(c1, y, true);
                    if (ex & 2) add_edge(c1, y, false);
                }
                pred[c2].clear();
                succ[c2].clear();
                gone[c2] = 1;
                ++nfold;
                folded = true;
                break;
            }
            if (!folded) break;
        }
    }
    if (!nfold) return 0;
    std::vector<int> inew(ni, -1);
    std::vector<Instr> instrs;
    for (int i = 0; i < ni; ++i)
        if (!gone[i]) { inew[i] = (int)instrs.size(); instrs.push_back(d.instrs[i]); }
    for (auto& X : d.xfers) {
        X.send_instr = inew[X.send_instr];
        X.recv_instr = inew[X.recv_instr];
    }
    std::vector<Dep> deps;
    for (int a = 0; a < ni; ++a) {
        if (gone[a]) continue;
        for (int b : succ[a]) {
            if (gone[b]) continue;
            auto it = exact.find({a, b});
            if (it == exact.end()) continue;   // a transfer edge
            if (it->second & 1) deps.push_back(Dep{inew[a], inew[b], true});
            if (it->second & 2) deps.push_back(Dep{inew[a], inew[b], false});
        }
    }
    d.instrs = std::move(instrs);
    d.deps = std::move(deps);
    return nfold;
}

// Reduction chains (after direct transport): a send or recv-reduce-send X
// whose slot feeds a receive-reduce Y (recv-reduce-send, -copy, or
// -copy-send) is run as one step by X's threadblock, which reads Y's local
// operand itself and adds it after X's sum (the chain's order, each sum
// rounded to the element type): send + rrs -> CCL_I_RSEND, send + rrc ->
// CCL_I_REDUCE, send + rrcs -> CCL_I_RCSEND, rrs + rrs / rrc / rrcs ->
// CCL_I_RRS3 / RRC3 / RRCS3 (Y's local operand held in the source range).
// The slot between them goes (2 bytes per element byte) and so does a hop;
// the folded step sends on where Y sent (a link two ranks ahead in a
// ring).  Pairs form in dependency order from each chain's head; a pair
// whose merged dependencies would close a cycle is left alone.
int fold_reduce_chains(ccl_schedule& d)
{
    const int ni = (int)d.instrs.size();
    std::vector<std::set<int>> succ(ni), pred(ni);
    std::map<std::pair<int, int>, int> exact;   // dependency edges: bit 0 exact, bit 1 not
    auto add_dep = [&](int a, int b, int bits) {
        if (a == b || !bits) return;
        succ[a].insert(b);
        pred[b].insert(a);
        exact[{a, b}] |= bits;
    };
    for (const Dep& e : d.deps) add_dep(e.from, e.to, e.exact ? 1 : 2);
    auto add_xfer_edge = [&](int a, int b) {
        if (a < 0 || b < 0) return;
        succ[a].insert(b);
        pred[b].insert(a);
    };
    for (const Xfer& X : d.xfers) add_xfer_edge(X.send_instr, X.recv_instr);
    std::vector<int> indeg(ni), order;
    std::set<int> ready;
    for (int i = 0; i < ni; ++i)
        if ((indeg[i] = (int)pred[i].size()) == 0) ready.insert(i);
    while (!ready.empty()) {
        const int i = *ready.begin();
        ready.erase(ready.begin());
        order.push_back(i);
        for (int j : succ[i])
            if (--indeg[j] == 0) ready.insert(j);
    }
    if ((int)order.size() != ni) return 0;
    std::vector<char> gone(ni, 0), merged(ni, 0), xgone(d.xfers.size(), 0);
    std::vector<int> mark(ni, -1);
    int nfold = 0, epoch = 0;
    for (int c1 : order) {
        if (gone[c1] || merged[c1]) continue;
        const Instr& X = d.instrs[c1];
        if ((X.kind != CCL_I_SEND && X.kind != CCL_I_RRS) || X.xfer_out < 0) continue;
        const int x = X.xfer_out;
        const int c2 = d.xfers[x].recv_instr;
        if (c2 < 0 || gone[c2] || merged[c2]) continue;
        const Instr& Y = d.instrs[c2];
        if (Y.kind != CCL_I_RRS && Y.kind != CCL_I_RRC && Y.kind != CCL_I_RRCS) continue;
        if (Y.count != X.count || !Y.loc.valid() || (X.kind == CCL_I_SEND && !X.src.valid())) continue;
        // everything else Y waits for must be able to come before X
        std::vector<int> stack{c1};
        bool cycle = false;
        mark[c1] = ++epoch;
        while (!stack.empty() && !cycle) {
            const int v = stack.back();
            stack.pop_back();
            for (int w : succ[v]) {
                if (w == c2 || mark[w] == epoch) continue;
                if (pred[c2].count(w)) { cycle = true; break; }
                mark[w] = epoch;
                stack.push_back(w);
            }
        }
        if (cycle) continue;
        Instr F = X;
        if (X.kind == CCL_I_SEND) {
            F.loc = Y.loc;
            F.kind = Y.kind == CCL_I_RRS ? CCL_I_RSEND : Y.kind == CCL_I_RRC ? CCL_I_REDUCE : CCL_I_RCSEND;
        } else {
            F.src = Y.loc;
            F.kind = Y.kind == CCL_I_RRS ? CCL_I_RRS3 : Y.kind == CCL_I_RRC ? CCL_I_RRC3 : CCL_I_RRCS3;
        }
        F.dst = Y.dst;
        F.xfer_out = Y.xfer_out;
        if (F.xfer_out >= 0) {
            d.xfers[F.xfer_out].send_instr = c1;
            d.xfers[F.xfer_out].src_rank = X.rank;
        }
        xgone[x] = 1;
        d.instrs[c1] = F;
        // c1 takes over c2's edges
        for (int w : std::vector<int>(pred[c2].begin(), pred[c2].end())) {
            auto it = exact.find({w, c2});
            const int bits = it == exact.end() ? 0 : it->second;
            succ[w].erase(c2);
            if (w != c1) add_dep(w, c1, bits);
        }
        for (int y : std::vector<int>(succ[c2].begin(), succ[c2].end())) {
            auto it = exact.find({c2, y});
            pred[y].erase(c2);
            if (it == exact.end()) add_xfer_edge(c1, y);   // the transfer c2 sent
            else add_dep(c1, y, it->second);
        }
        pred[c2].clear();
        succ[c2].clear();
        gone[c2] = 1;
        merged[c1] = 1;
        ++nfold;
    }
    if (!nfold) return 0;
    std::vector<int> inew(ni, -1);
    std::vector<Instr> instrs;
    for (int i = 0; i < ni; ++i)
        if (!gone[i]) { inew[i] = (int)instrs.size(); instrs.push_back(d.instrs[i]); }
    std::vector<int> xnew(d.xfers.size(), -1);
    std::vector<Xfer> xfers;
    for (size_t x = 0; x < d.xfers.size(); ++x)
        if (!xgone[x]) { xnew[x] = (int)xfers.size(); xfers.push_back(d.xfers[x]); }
    for (auto& I : instrs) {
        if (I.xfer_in >= 0) I.xfer_in = xnew[I.xfer_in];
        if (I.xfer_out >= 0) I.xfer_out = xnew[I.xfer_out];
    }
    for (auto& X : xfers) {
        X.send_instr = inew[X.send_instr];
        X.recv_instr = inew[X.recv_instr];
    }
    std::vector<Dep> deps;
    for (const auto& kv : exact) {
        const int a = kv.first.first, b = kv.first.second;
        if (gone[a] || gone[b] || !succ[a].count(b)) continue;
        if (kv.second & 1) deps.push_back(Dep{inew[a], inew[b], true});
        if (kv.second & 2) deps.push_back(Dep{inew[a], inew[b], false});
    }
    d.instrs = std::move(instrs);
    d.xfers = std::move(xfers);
    d.deps = std::move(deps);
    return nfold;
}

namespace {

ccl_status_t build_plan_one(const ccl_schedule& s_in, int64_t ce, int32_t dtype, const ccl_plan_opts_t& o,
                            PlanImage* img, int fold)
{
    if (ce <= 0) return fail(CCL_ERR_INVALID_ARG, "chunk_elems must be positive");
    if (dtype < CCL_F32 || dtype > CCL_I32) return fail(CCL_ERR_INVALID_ARG, "unknown dtype");
    if (o.channels < 1 || o.channels > 256) return fail(CCL_ERR_INVALID_ARG, "channels must be in 1..256");
    if (o.nthreads < 128 || o.nthreads > 1024 || o.nthreads % 32)
        return fail(CCL_ERR_INVALID_ARG, "nthreads must be a multiple of 32 in 128..1024");
    if (o.bulk != 0 && o.bulk != 1) return fail(CCL_ERR_INVALID_ARG, "bulk must be 0 or 1");
    if (o.engine != CCL_ENGINE_PIPELINED && o.engine != CCL_ENGINE_SEQUENTIAL)
        return fail(CCL_ERR_INVALID_ARG, "engine must be CCL_ENGINE_PIPELINED or CCL_ENGINE_SEQUENTIAL");
    if (o.cluster != 0 && o.cluster != 1 && o.cluster != 2 && o.cluster != 4 && o.cluster != 8)
        return fail(CCL_ERR_INVALID_ARG, "cluster must be 0, 1, 2, 4 or 8");
    if (o.cluster > 1 && o.engine != CCL_ENGINE_SEQUENTIAL)
        return fail(CCL_ERR_UNSUPPORTED, "clusters of CTAs run the sequential engine only");
    if (o.channel_scaling != 0 && o.channel_scaling != 1)
        return fail(CCL_ERR_INVALID_ARG, "channel_scaling must be 0 or 1");
    if (o.tile_bytes < 16 || o.tile_bytes % 16 || o.tile_bytes > 65536)
        return fail(CCL_ERR_INVALID_ARG, "tile_bytes must be a multiple of 16 in 16..65536");
    if (o.slot_bytes < 16 || o.slot_bytes % 16) return fail(CCL_ERR_INVALID_ARG, "slot_bytes must be a positive multiple of 16");
    if (o.fifo_slots < 2 || o.fifo_slots > 64) return fail(CCL_ERR_INVALID_ARG, "fifo_slots must be in 2..64");
    if (o.microbatches < 0 || o.microbatches > 65536) return fail(CCL_ERR_INVALID_ARG, "microbatches out of range");
    if (o.scheduler != CCL_SCHED_RR && o.scheduler != CCL_SCHED_HPDS) return fail(CCL_ERR_INVALID_ARG, "unknown scheduler");
    if (o.tb_alloc != CCL_TB_CONNECTION && o.tb_alloc != CCL_TB_PACKED && o.tb_alloc != CCL_TB_BALANCED)
        return fail(CCL_ERR_INVALID_ARG, "unknown tb_alloc");
    if (o.tb_budget < 0) return fail(CCL_ERR_INVALID_ARG, "tb_budget must not be negative");
    if (o.mb_order < CCL_MB_AUTO || o.mb_order > CCL_MB_SEGMENT) return fail(CCL_ERR_INVALID_ARG, "unknown mb_order");
    if (o.mb_window < 0 || o.mb_window > 65536) return fail(CCL_ERR_INVALID_ARG, "mb_window out of range");
    if (o.protocol != CCL_PROTO_SIMPLE && o.protocol != CCL_PROTO_LL) return fail(CCL_ERR_INVALID_ARG, "unknown protocol");
    if (o.protocol == CCL_PROTO_LL && (ce * esize_of(dtype)) % 16)
        return fail(CCL_ERR_UNSUPPORTED, "the LL protocol needs chunks of a multiple of 16 bytes");
    if (o.timeout_ms <= 0) return fail(CCL_ERR_INVALID_ARG, "timeout_ms must be positive");
    if (o.fold < 0 || o.fold > 15) return fail(CCL_ERR_INVALID_ARG, "fold must be in 0..15");

    if (o.link_mode != CCL_LINK_FIFO && o.link_mode != CCL_LINK_DIRECT)
        return fail(CCL_ERR_INVALID_ARG, "unknown link_mode");
    int ndirect = 0;
    ccl_schedule s = s_in;
    if (o.link_mode == CCL_LINK_DIRECT) {
        // reduction chains first (a recv-reduce-copy-send taken into a pair
        // keeps its receive on a FIFO; the LL slots' path takes no third
        // operand), then plain transfers and receive folds, then copy chains
        if ((fold & 4) && o.protocol != CCL_PROTO_LL) fold_reduce_chains(s);
        s = direct_transport(s, &ndirect, (fold & 1) != 0);
        // copy chains: two hops per step (bit 1), three (bit 3)
        if (fold & 10) fold_copy_chains(s, (fold & 8) ? 3 : 2);
    }
    const int es = esize_of(dtype);
    Timeline tl;
    ccl_status_t st = build_timeline(s, o.scheduler, &tl);
    if (st != CCL_OK) return st;

    TBList conn;
    std::vector<int> conn_rank;
    allocate_connection(s, tl, &conn, &conn_rank);
    TBList packed = conn;
    std::vector<int> packed_rank = conn_rank;
    if (o.tb_alloc == CCL_TB_PACKED || o.tb_alloc == CCL_TB_BALANCED) pack_state_based(s, tl, &packed, &packed_rank);
    if (o.tb_alloc == CCL_TB_BALANCED) {
        const int budget = o.tb_budget > 0 ? o.tb_budget : 256;
        balance_linkfree(s, tl, &packed, &packed_rank, std::max(1, budget / std::max(1, o.channels)));
    }

    // micro-batch candidates
    int64_t max_slots = 1;
    int64_t max_per_ch = 0;   // elements of the largest linked channel range
    const std::vector<int> pcs = channel_counts(s, o.channels, o.channel_scaling);
    for (size_t i = 0; i < s.instrs.size(); ++i) {
        const Instr& I = s.instrs[i];
        if (I.xfer_in < 0 && I.xfer_out < 0) continue;
        int64_t n = I.count * ce;
        int64_t per_ch = (n + pcs[i] - 1) / pcs[i];
        max_per_ch = std::max(max_per_ch, per_ch);
        max_slots = std::max<int64_t>(max_slots, (per_ch * es + o.slot_bytes - 1) / o.slot_bytes);
    }
    int64_t half = std::max(1, o.fifo_slots / 2);
    int m_small = (int)std::min<int64_t>(4096, (max_slots + half - 1) / half);
    std::vector<int> ms;
    // small pieces first: instructions sharing a threadblock then interleave
    // piece by piece instead of running one after the other
    if (o.microbatches > 0) ms.push_back(o.microbatches);
    else { ms.push_back(m_small); if (m_small > 1) ms.push_back(1); }
    std::vector<int> orders;
    if (o.mb_order == CCL_MB_AUTO) orders = {CCL_MB_ALGO, CCL_MB_SEGMENT, CCL_MB_TASK};
    else orders = {o.mb_order};
    std::vector<int> allocs;
    if (o.tb_alloc == CCL_TB_PACKED || o.tb_alloc == CCL_TB_BALANCED) allocs = {CCL_TB_PACKED, CCL_TB_CONNECTION};
    else allocs = {CCL_TB_CONNECTION};

    std::string first_why;
    for (int alloc : allocs) {
        const TBList& tbs = alloc == CCL_TB_PACKED ? packed : conn;
        const std::vector<int>& tr = alloc == CCL_TB_PACKED ? packed_rank : conn_rank;
        for (int m : ms) {
            std::vector<int> wins;
            if (o.mb_window > 0) wins.push_back(std::min(m, o.mb_window));
            else {
                // double buffering: a window's slots and the next window's
                // fit in the FIFO together, so neighbours do not run in
                // lockstep (a piece takes ceil(per-channel range / m) bytes
                // in slots)
                const int64_t piece_slots =
                    std::max<int64_t>(1, (max_per_ch + m - 1) / m * es / o.slot_bytes +
                                             ((max_per_ch + m - 1) / m * es % o.slot_bytes ? 1 : 0));
                const int w = (int)std::max<int64_t>(1, std::min<int64_t>(m, o.fifo_slots / (2 * piece_slots)));
                wins.push_back(w);
                if (w > 1) wins.push_back(1);
            }
            for (int order : orders) for (int window : wins) {
                PlanImage cand;
                st = build_image(s, tl, tbs, tr, ce, dtype, o, m, order, window, &cand);
                std::string why;
                if (st == CCL_ERR_DEADLOCK) {
                    if (first_why.empty()) first_why = ccl_last_error_detail();
                    continue;
                }
                if (st != CCL_OK) return st;
                if (log_level() >= 2) dump_programs(s, tl, tbs, tr, m, order);
                if (simulate_plan(cand, &why)) {
                    *img = std::move(cand);
                    img->ntb_connection = (int)conn.size() * o.channels;
                    img->channel_scaling = o.channel_scaling;
                    goto done;
                }
                if (first_why.empty())
                    first_why = "m=" + std::to_string(m) + " order=" + std::to_string(order) +
                                " window=" + std::to_string(window) + ": " + why;
            }
        }
    }
    return fail(CCL_ERR_DEADLOCK, "threadblock programs cannot finish with " + std::to_string(o.fifo_slots) +
                                      " FIFO slots of " + std::to_string(o.slot_bytes) + " bytes (" + first_why + ")");
done:
    img->ndirect = ndirect;
    img->cluster = o.cluster > 1 ? o.cluster : 1;
    if (log_level() >= 1) {
        size_t drains = 0, waiting = 0;
        for (const DStep& d : img->steps) {
            drains += d.drain >= 0;
            waiting += d.dep_count > 0;
        }
        std::fprintf(stderr,
                     "[ccl] plan: %d threadblocks, %zu steps, m=%d order=%d window=%d, %zu steps follow an earlier "
                     "step of their threadblock, %zu steps wait on %zu counters\n",
                     img->ntb, img->steps.size(), img->m, img->mb_order, img->mb_window, drains, waiting,
                     img->deps.size());
    }
    // byte accounting of the source program
    {
        std::vector<std::vector<char>> rd(s.nranks, std::vector<char>(std::max(1, s.nchunks[0]), 0));
        std::vector<std::vector<char>> wr(s.nranks, std::vector<char>(std::max(1, s.nchunks[1]), 0));
        for (const ccl_op_t& op : s.ops) {
            if (op.src_buf == CCL_BUF_IN)
                for (int k = 0; k < op.count; ++k) rd[op.src_rank][op.src_off + k] = 1;
            if (op.dst_buf == CCL_BUF_OUT)
                for (int k = 0; k < op.count; ++k) wr[op.dst_rank][op.dst_off + k] = 1;
        }
        int64_t c = 0;
        for (int r = 0; r < s.nranks; ++r) {
            for (char v : rd[r]) c += v;
            for (char v : wr[r]) c += v;
        }
        img->min_bytes = c * ce * es;
    }
    img->in_elems = (int64_t)s.nchunks[0] * ce;
    img->out_elems = (int64_t)s.nchunks[1] * ce;
    img->scratch_elems = (int64_t)s.nchunks[2] * ce;
    {
        double R = s.nranks;
        int64_t in_b = img->in_elems * es, out_b = img->out_elems * es;
        switch (s.builtin) {
        case CCL_RING_ALLREDUCE:
        case CCL_HIER_ALLREDUCE: img->data_bytes_per_rank = in_b; img->busbw_factor = 2.0 * (R - 1) / R; break;
        case CCL_RING_ALLGATHER: img->data_bytes_per_rank = out_b; img->busbw_factor = (R - 1) / R; break;
        case CCL_RING_REDUCESCATTER: img->data_bytes_per_rank = in_b; img->busbw_factor = (R - 1) / R; break;
        case CCL_ALLTOALL_2PHASE: img->data_bytes_per_rank = in_b; img->busbw_factor = (R - 1) / R; break;
        case CCL_ALLTOALLV: img->data_bytes_per_rank = in_b; img->busbw_factor = (R - 1) / R; break;
        case CCL_ALLTONEXT: img->data_bytes_per_rank = in_b; img->busbw_factor = 1.0; break;
        default: img->data_bytes_per_rank = in_b; img->busbw_factor = 0.0; break;
        }
    }
    img->fuse = s.fuse;
    return CCL_OK;
}

}  // namespace

// Fusion moves a send into the step that produces its data, so a fused
// program keeps more transfers in flight on a link than its unfused form and
// can need more FIFO slots, or a task order the timeline cannot build, where
// the unfused program plans.  Both compute the same values, so a fused
// schedule that cannot be planned with the given options is planned from the
// same program compiled with less fusion (full -> copy receives unchained ->
// none); the plan reports the mode it used.
ccl_status_t build_plan(const ccl_schedule& s, int64_t ce, int32_t dtype, const ccl_plan_opts_t& o,
                        PlanImage* img)
{
    // with direct transport, the plain receive of a copy-send or a
    // recv-reduce-copy-send is folded into its sender first (one pass
    // writes both destinations); where the folds make the timeline cyclic
    // or the threadblocks deadlock, they are given up a kind at a time:
    // three-hop copy chains first (keeping two hops), then reduction
    // chains, then both, then all copy chains, then the receive folds
    const int fold = o.link_mode == CCL_LINK_DIRECT ? o.fold : 0;
    auto plan_one = [&](const ccl_schedule& x) {
        ccl_status_t r = build_plan_one(x, ce, dtype, o, img, fold);
        if (fold && (r == CCL_ERR_CYCLE || r == CCL_ERR_DEADLOCK)) {
            const std::string why = ccl_last_error_detail();
            const int two = (fold & ~8) | (fold & 8 ? 2 : 0);   // three hops -> two
            int tried[7] = {fold}, ntried = 1;
            for (int f : {two, fold & ~4, two & ~4, fold & 5, fold & 1, 0}) {
                if (std::find(tried, tried + ntried, f) != tried + ntried) continue;
                tried[ntried++] = f;
                if (build_plan_one(x, ce, dtype, o, img, f) == CCL_OK) return CCL_OK;
            }
            fail(r, why);
        }
        return r;
    };
    ccl_status_t st = plan_one(s);
    if ((st != CCL_ERR_CYCLE && st != CCL_ERR_DEADLOCK) || s.fuse == CCL_FUSE_NONE) return st;
    const std::string first = ccl_last_error_detail();
    for (int mode : {CCL_FUSE_NOCHAIN, CCL_FUSE_NONE}) {
        if (mode == s.fuse || (s.fuse == CCL_FUSE_NOCHAIN && mode != CCL_FUSE_NONE)) continue;
        ccl_schedule less;
        if (compile_program(s.ops.data(), (int)s.ops.size(), s.nranks, s.nchunks, mode, &less) != CCL_OK) break;
        less.builtin = s.builtin;
        less.group_size = s.group_size;
        if (plan_one(less) == CCL_OK) {
            if (log_level() >= 1)
                std::fprintf(stderr, "[ccl] fused schedule did not plan (%s); planned with fusion mode %d\n",
                             first.c_str(), mode);
            return CCL_OK;
        }
    }
    return fail(st, first);
}

}  // namespace ccl
