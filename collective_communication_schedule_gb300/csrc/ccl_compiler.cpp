// Host compiler: chunk program -> fused per-rank instructions.
//
// MSCCLang report, §III.1 "system design": the compiler traces the chunk
// program into a dependency DAG, lowers every cross-rank operation into a
// send on the source rank and a receive (or receive-reduce) on the
// destination rank, and fuses adjacent instructions into compound ones such
// as recv-reduce-copy-send so that memory traffic and synchronisation drop.
//
// Implementation: every operation becomes one or two "halves" carrying the
// ranges they read and write on their rank.  A value analysis over each
// rank's halves (in program order) finds, for the value a half writes, the
// later halves that read exactly that range before it is overwritten, and
// whether it survives to the end in an input/output buffer.  Three rewrite
// rules are applied until nothing changes:
//   R1 copy propagation into a reduce: dst := src ; dst := dst (+) x
//      becomes dst := src (+) x when the copied value has no other reader;
//   R2 copy propagation into a send: a send of a freshly copied value reads
//      the copy's source instead (the copy disappears when its value is dead
//      afterwards), or copy and send merge into copy-send;
//   R3 receive chaining: a received (or received-and-reduced) value that is
//      sent on becomes recv-copy-send / recv-reduce-copy-send, and the local
//      write is dropped when nothing else reads the value (recv-send,
//      recv-reduce-send).
// Each rule only moves a send earlier to the position of the instruction
// that produced its data, or re-routes a read to an unchanged equal value, so
// the program's results are unchanged.
#include <algorithm>
#include <map>
#include <string>

#include "ccl_internal.h"

namespace ccl {

int64_t kind_bytes_factor(int kind)
{
    switch (kind) {
    case CCL_I_COPY: return 2;
    case CCL_I_REDUCE: return 3;
    case CCL_I_SEND: return 2;
    case CCL_I_RECV: return 2;
    case CCL_I_RRC: return 3;
    case CCL_I_RCS: return 3;
    case CCL_I_FWD: return 2;
    case CCL_I_RRS: return 3;
    case CCL_I_RRCS: return 4;
    case CCL_I_COPY_SEND: return 3;
    case CCL_I_COPY2: return 3;
    case CCL_I_RRC2: return 4;
    case CCL_I_RRS3: return 4;
    case CCL_I_RRC3: return 4;
    case CCL_I_RRCS3: return 5;
    case CCL_I_RSEND: return 3;
    case CCL_I_RCSEND: return 4;
    case CCL_I_RRC3D: return 5;
    case CCL_I_REDUCE2: return 4;
    case CCL_I_COPY3: return 4;
    default: return 0;
    }
}

bool kind_reads_slot(int k)
{
    return k == CCL_I_RECV || k == CCL_I_RRC || k == CCL_I_RCS || k == CCL_I_FWD ||
           k == CCL_I_RRS || k == CCL_I_RRCS;
}
bool kind_writes_slot(int k)
{
    return k == CCL_I_SEND || k == CCL_I_RCS || k == CCL_I_FWD || k == CCL_I_RRS ||
           k == CCL_I_RRCS || k == CCL_I_COPY_SEND;
}
bool kind_is_reduce(int k)
{
    return k == CCL_I_REDUCE || k == CCL_I_RRC || k == CCL_I_RRS || k == CCL_I_RRCS;
}

namespace {

struct Half {
    bool alive = true;
    int rank = -1;
    int pos = 0;
    int recv_x = -1;          // transfer received
    bool recv_reduce = false; // received data is added to `loc`
    int send_x = -1;          // transfer sent
    bool local_reduce = false;// dst := loc (+) src on one rank
    Range src, loc, dst;
    int64_t count = 0;
};

bool pure_copy(const Half& h)
{
    return h.recv_x < 0 && h.send_x < 0 && !h.local_reduce && h.src.valid() && h.dst.valid();
}
bool send_only(const Half& h)
{
    return h.send_x >= 0 && h.recv_x < 0 && !h.local_reduce && !h.dst.valid() && h.src.valid();
}

struct ValueInfo {
    std::vector<int> consumers;  // halves reading exactly the written range
    bool escaping = false;       // read or overwritten partially
    bool killed = false;         // overwritten exactly
    bool liveout = false;        // still present at the end in an in/out buffer
};

class Fuser {
public:
    bool chain_copies = true;  // R3 also chains receives that only copy
    std::vector<int> xfer_dst; // receiving rank of every transfer
    std::vector<Half> h;
    std::vector<std::vector<int>> per_rank;  // indices into h, sorted by pos

    std::vector<std::vector<int>> per_pos;   // alive halves at each program position
    std::vector<int> sender;                 // alive half that sends each transfer

    void index(int nranks)
    {
        per_rank.assign(nranks, {});
        int npos = 0;
        for (const Half& x : h) npos = std::max(npos, x.pos + 1);
        per_pos.assign(npos, {});
        sender.assign(xfer_dst.size(), -1);
        for (int i = 0; i < (int)h.size(); ++i) {
            if (!h[i].alive) continue;
            per_rank[h[i].rank].push_back(i);
            per_pos[h[i].pos].push_back(i);
            if (h[i].send_x >= 0) sender[h[i].send_x] = i;
        }
        for (auto& v : per_rank)
            std::sort(v.begin(), v.end(), [&](int a, int b) { return h[a].pos < h[b].pos; });
    }

    ValueInfo analyse(int w)
    {
        ValueInfo vi;
        const Range& D = h[w].dst;
        const auto& lst = per_rank[h[w].rank];
        bool after = false;
        for (int x : lst) {
            if (x == w) { after = true; continue; }
            if (!after || !h[x].alive) continue;
            bool cons = false;
            for (const Range* r : {&h[x].src, &h[x].loc}) {
                if (!r->overlaps(D)) continue;
                if (r->same(D)) cons = true; else vi.escaping = true;
            }
            if (cons) vi.consumers.push_back(x);
            if (h[x].dst.overlaps(D)) {
                if (h[x].dst.same(D)) vi.killed = true; else vi.escaping = true;
                break;
            }
        }
        vi.liveout = vi.escaping || (!vi.killed && D.buf != CCL_BUF_SCRATCH);
        return vi;
    }

    // no alive half on `rank` with position in (p0, p1] writes a range
    // overlapping A
    bool unchanged(const Range& A, int rank, int p0, int p1)
    {
        for (int x : per_rank[rank]) {
            const Half& y = h[x];
            if (!y.alive || y.pos <= p0 || y.pos > p1) continue;
            if (y.dst.overlaps(A)) return false;
        }
        return true;
    }

    // Moving X's send up to W (R2, R3) changes the order of the sends on the
    // link W.rank -> dst.  The planner orders a threadblock's steps by their
    // dependencies, so that is harmless unless a send to dst between the two
    // positions must itself follow W: then the moved send would overtake it
    // on the link while its receiver still takes them in program order.
    // True when no alive half of W's rank strictly between W and X depends
    // on W and sends to dst.  "Depends" is the closure of two edges, followed
    // over every rank: a later half of the same rank that touches a range
    // the other half wrote (or writes a range it read), and the receiving
    // half of a transfer whose sending half depends on W -- so a chain that
    // leaves W's rank through a transfer and comes back counts too.  Both
    // edges only go forward in program position, so one pass over the
    // positions between W and X finds the closure.
    bool can_move_send_up(int w, int xpos, int dst)
    {
        const Half& W = h[w];
        auto reads = [](const Half& a, const Range& r) { return a.src.overlaps(r) || a.loc.overlaps(r); };
        auto touches = [&](const Half& y, const Half& z) {   // y later than z on z's rank
            return (z.dst.valid() && (reads(y, z.dst) || y.dst.overlaps(z.dst))) ||
                   (y.dst.valid() && reads(z, y.dst));
        };
        std::vector<char> is_dep(h.size(), 0);
        std::vector<std::vector<int>> dep_of_rank(per_rank.size());
        is_dep[w] = 1;
        dep_of_rank[W.rank].push_back(w);
        for (int p = W.pos; p < xpos && p < (int)per_pos.size(); ++p) {
            // a position holds one operation: its send half (possibly moved
            // into an earlier half) and its receive half; two rounds let a
            // receive see its sender's verdict at the same position
            for (int round = 0; round < 2; ++round) {
                for (int x : per_pos[p]) {
                    if (is_dep[x]) continue;
                    const Half& y = h[x];
                    bool d = y.recv_x >= 0 && sender[y.recv_x] >= 0 && is_dep[sender[y.recv_x]];
                    for (size_t k = 0; !d && k < dep_of_rank[y.rank].size(); ++k) {
                        const Half& z = h[dep_of_rank[y.rank][k]];
                        d = z.pos < y.pos && touches(y, z);
                    }
                    if (!d) continue;
                    if (y.rank == W.rank && y.pos > W.pos && y.send_x >= 0 && xfer_dst[y.send_x] == dst)
                        return false;
                    is_dep[x] = 1;
                    dep_of_rank[y.rank].push_back(x);
                }
            }
        }
        return true;
    }

    bool step()
    {
        for (auto& lst : per_rank) {
            for (int w : lst) {
                Half& W = h[w];
                if (!W.alive || !W.dst.valid()) continue;
                ValueInfo vi = analyse(w);
                // R1: copy propagation into a reduce
                if (pure_copy(W) && !vi.escaping && vi.consumers.size() == 1) {
                    Half& X = h[vi.consumers[0]];
                    if (X.loc.same(W.dst) && !X.src.same(W.dst) &&
                        unchanged(W.src, W.rank, W.pos, X.pos)) {
                        X.loc = W.src;
                        bool dead = !vi.liveout;
                        if (dead) W.alive = false;
                        return true;
                    }
                }
                // R2: copy propagation into a send
                if (pure_copy(W)) {
                    for (int xi : vi.consumers) {
                        Half& X = h[xi];
                        if (!send_only(X) || !X.src.same(W.dst)) continue;
                        if (!unchanged(W.src, W.rank, W.pos, X.pos)) continue;
                        if (vi.consumers.size() == 1 && !vi.liveout) {
                            X.src = W.src;
                            W.alive = false;
                        } else {
                            // the send moves up to W's position
                            if (!can_move_send_up(w, X.pos, xfer_dst[X.send_x])) continue;
                            W.send_x = X.send_x;
                            X.alive = false;
                        }
                        return true;
                    }
                }
                // R3: receive chaining
                if (W.recv_x >= 0 && W.send_x < 0 && (chain_copies || W.recv_reduce)) {
                    for (int xi : vi.consumers) {
                        Half& X = h[xi];
                        if (!send_only(X) || !X.src.same(W.dst)) continue;
                        // the send moves up to W's position
                        if (!can_move_send_up(w, X.pos, xfer_dst[X.send_x])) continue;
                        W.send_x = X.send_x;
                        X.alive = false;
                        if (vi.consumers.size() == 1 && !vi.liveout) W.dst = Range();
                        return true;
                    }
                }
            }
        }
        return false;
    }
};

}  // namespace

int fuse_mode(uint32_t flags)
{
    if (flags & CCL_FLAG_NOFUSE) return CCL_FUSE_NONE;
    return (flags & CCL_FLAG_NOCHAIN_COPIES) ? CCL_FUSE_NOCHAIN : CCL_FUSE_FULL;
}

namespace {

int kind_of(const Half& x)
{
    if (x.recv_x < 0 && x.send_x < 0) return x.local_reduce ? CCL_I_REDUCE : CCL_I_COPY;
    if (x.recv_x < 0) return x.dst.valid() ? CCL_I_COPY_SEND : CCL_I_SEND;
    if (x.send_x < 0) return x.recv_reduce ? CCL_I_RRC : CCL_I_RECV;
    if (x.recv_reduce) return x.dst.valid() ? CCL_I_RRCS : CCL_I_RRS;
    return x.dst.valid() ? CCL_I_RCS : CCL_I_FWD;
}

}  // namespace

ccl_status_t compile_program(const ccl_op_t* ops, int nops, int nranks, const int32_t nchunks[3],
                             int fuse, ccl_schedule* s)
{
    if (nranks < 1 || nranks > CCL_MAX_RANKS)
        return fail(CCL_ERR_INVALID_ARG, "nranks must be in 1.." + std::to_string(CCL_MAX_RANKS));
    if (nops < 0 || (nops > 0 && !ops)) return fail(CCL_ERR_INVALID_ARG, "bad op array");
    for (int b = 0; b < 3; ++b)
        if (nchunks[b] < 0) return fail(CCL_ERR_INVALID_ARG, "negative chunk count");
    for (int i = 0; i < nops; ++i) {
        const ccl_op_t& o = ops[i];
        std::string where = "op " + std::to_string(i) + ": ";
        if (o.op != CCL_OP_COPY && o.op != CCL_OP_REDUCE)
            return fail(CCL_ERR_INVALID_ARG, where + "unknown opcode");
        if (o.src_rank < 0 || o.src_rank >= nranks || o.dst_rank < 0 || o.dst_rank >= nranks)
            return fail(CCL_ERR_INVALID_ARG, where + "rank out of range");
        if (o.src_buf < 0 || o.src_buf > 2 || o.dst_buf < 0 || o.dst_buf > 2)
            return fail(CCL_ERR_INVALID_ARG, where + "unknown buffer kind");
        if (o.count <= 0) return fail(CCL_ERR_INVALID_ARG, where + "count must be positive");
        if (o.src_off < 0 || (int64_t)o.src_off + o.count > nchunks[o.src_buf] || o.dst_off < 0 ||
            (int64_t)o.dst_off + o.count > nchunks[o.dst_buf])
            return fail(CCL_ERR_INVALID_ARG, where + "chunk range outside the buffer");
        if (o.src_rank == o.dst_rank && o.src_buf == o.dst_buf && o.src_off < o.dst_off + o.count &&
            o.dst_off < o.src_off + o.count)
            return fail(CCL_ERR_INVALID_ARG, where + "source and destination overlap");
    }

    s->nranks = nranks;
    s->fuse = fuse;
    for (int b = 0; b < 3; ++b) s->nchunks[b] = nchunks[b];
    s->ops.assign(ops, ops + nops);

    // ---- lowering: one or two halves per operation
    Fuser F;
    std::vector<Xfer> xf;
    for (int i = 0; i < nops; ++i) {
        const ccl_op_t& o = ops[i];
        Range S{o.src_rank, o.src_buf, o.src_off, o.count};
        Range D{o.dst_rank, o.dst_buf, o.dst_off, o.count};
        if (o.src_rank == o.dst_rank) {
            Half x;
            x.rank = o.src_rank; x.pos = i; x.count = o.count;
            x.src = S; x.dst = D;
            if (o.op == CCL_OP_REDUCE) { x.local_reduce = true; x.loc = D; }
            F.h.push_back(x);
        } else {
            int id = (int)xf.size();
            Xfer t;
            t.src_rank = o.src_rank; t.dst_rank = o.dst_rank; t.count = o.count;
            t.chunk_id = o.src_off;
            t.op_index = i;
            xf.push_back(t);
            F.xfer_dst.push_back(o.dst_rank);
            Half snd;
            snd.rank = o.src_rank; snd.pos = i; snd.count = o.count; snd.send_x = id; snd.src = S;
            Half rcv;
            rcv.rank = o.dst_rank; rcv.pos = i; rcv.count = o.count; rcv.recv_x = id; rcv.dst = D;
            if (o.op == CCL_OP_REDUCE) { rcv.recv_reduce = true; rcv.loc = D; }
            F.h.push_back(snd);
            F.h.push_back(rcv);
        }
    }
    F.index(nranks);
    F.chain_copies = fuse != CCL_FUSE_NOCHAIN;
    if (fuse != CCL_FUSE_NONE) {
        int guard = 0;
        while (F.step()) {
            F.index(nranks);
            if (++guard > 10 * (int)F.h.size() + 100)
                return fail(CCL_ERR_INTERNAL, "fusion did not converge");
        }
    }

    // ---- emit instructions sorted by (rank, position)
    s->instrs.clear();
    for (int r = 0; r < nranks; ++r) {
        for (int idx : F.per_rank[r]) {
            const Half& x = F.h[idx];
            if (!x.alive) continue;
            Instr in;
            in.kind = kind_of(x);
            in.rank = x.rank;
            in.src = x.src; in.loc = x.loc; in.dst = x.dst;
            in.count = x.count;
            in.xfer_in = x.recv_x; in.xfer_out = x.send_x;
            in.position = x.pos;
            // a receive-reduce whose local operand is gone cannot happen
            if (kind_is_reduce(in.kind) && !in.loc.valid())
                return fail(CCL_ERR_INTERNAL, "reduce without local operand");
            int id = (int)s->instrs.size();
            if (in.xfer_in >= 0) xf[in.xfer_in].recv_instr = id;
            if (in.xfer_out >= 0) xf[in.xfer_out].send_instr = id;
            s->instrs.push_back(in);
        }
    }
    for (auto& t : xf)
        if (t.send_instr < 0 || t.recv_instr < 0)
            return fail(CCL_ERR_INTERNAL, "transfer lost an end during fusion");
    s->xfers = xf;

    // ---- same-rank buffer hazards between the fused instructions
    s->deps.clear();
    int n = (int)s->instrs.size();
    int i0 = 0;
    while (i0 < n) {
        int i1 = i0;
        while (i1 < n && s->instrs[i1].rank == s->instrs[i0].rank) ++i1;
        for (int j = i0; j < i1; ++j) {
            const Instr& b = s->instrs[j];
            for (int i = i0; i < j; ++i) {
                const Instr& a = s->instrs[i];
                bool hz = false, exact = true;
                auto chk = [&](const Range& x, const Range& y) {
                    if (x.overlaps(y)) { hz = true; if (!x.same(y)) exact = false; }
                };
                // RAW, WAR, WAW
                chk(a.dst, b.src); chk(a.dst, b.loc);
                chk(a.src, b.dst); chk(a.loc, b.dst);
                chk(a.dst, b.dst);
                if (hz) s->deps.push_back(Dep{i, j, exact});
            }
        }
        i0 = i1;
    }
    return CCL_OK;
}

}  // namespace ccl
