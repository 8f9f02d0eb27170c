// Kernels generated for single plans (ReSCCL report, §II.2 "lightweight
// kernel generation": code per rank x threadblock x pipeline instead of an
// instruction interpreter at run time).
//
// The generator turns every threadblock program of a plan into a device
// function whose code walks the program's segments, windows and micro-batch
// pieces in loops, one call per instruction and window.  The constants of
// each channel instruction -- kind, data type, buffers, element offsets,
// link slot and flag bases, dependency and signal counters, drain rule,
// cache hints -- are compiled into the generated module as read-only data;
// the piece of a micro-batch (the planner's 16-byte-granular split), its
// FIFO slot count and the sequence numbers on each link (running sums in the
// order the threadblock sends or receives) are computed where they are
// used, and each step runs the library's own seq_step / issue_step.  None
// of the plan's step records, link table or dependency lists is read at
// run time: a plan with a generated kernel uploads only its flags and FIFOs'
// state.
//
// Before it emits anything the generator replays those loops and formulas
// on the host and compares every step with the planner's record; a plan
// whose steps they do not reproduce (for example a receiver that takes a
// link's pieces in another order than its sender) is refused rather than
// approximated.
#include <cstdint>
#include <map>
#include <set>
#include <string>
#include <vector>

#include "ccl_plan.h"

namespace ccl {
namespace {

struct DepForm {
    std::vector<int> exact;   // counters waited with value mb + 1 at every piece
    std::vector<int> whole;   // counters waited with value m at piece 0
};

// per channel instruction of a threadblock: what its steps share
struct InstrForm {
    int ci = -1;
    int signal = -1;
    int flags = 0;
    DepForm deps;
    // drain: 0 none, 2 a fixed step, 3 a fixed distance back, 4 the same
    // micro-batch of another instruction of the threadblock (its step index
    // from that instruction's segment: base, instructions, window, position)
    int drain_kind = 0;
    int drain_dk = 0;
    int drain_const = -1;
    long long p_base = 0;
    int p_n = 0, p_w = 1, p_pos = 0;
};

// step index of micro-batch mb of the instruction at position pos of a
// segment starting at step base with n instructions in windows of w
long long seg_step(long long base, int n, int w, int pos, int mb, int m)
{
    const int w0 = mb / w * w;
    const int wl = std::min(m, w0 + w) - w0;
    return base + (long long)w0 * n + (long long)pos * wl + (mb - w0);
}

// the step a drain form names for step k (micro-batch mb)
long long drain_of(const InstrForm& f, int k, int mb, int m)
{
    switch (f.drain_kind) {
    case 2: return f.drain_const;
    case 3: return k - f.drain_dk;
    case 4: return seg_step(f.p_base, f.p_n, f.p_w, f.p_pos, mb, m);
    default: return -1;
    }
}

std::string lit(long long v) { return std::to_string(v) + "ll"; }


using DepSet = std::set<std::pair<int, long long>>;

DepSet step_deps(const PlanImage& img, const DStep& st)
{
    DepSet s;
    for (int k = 0; k < st.dep_count; ++k) {
        const DDep& d = img.deps[st.dep_begin + k];
        s.insert({d.counter, d.value});
    }
    return s;
}

DepSet form_deps(const DepForm& f, int mb, int m)
{
    std::map<int, long long> v;
    for (int c : f.exact) v[c] = mb + 1;
    if (mb == 0)
        for (int c : f.whole) v[c] = std::max<long long>(v.count(c) ? v[c] : 0, m);
    DepSet s;
    for (auto& e : v) s.insert({e.first, e.second});
    return s;
}

}  // namespace

std::string generate_plan_source(const PlanImage& img, int build, std::string* why)
{
    auto refuse = [&](const std::string& msg) {
        *why = msg;
        return std::string();
    };
    if (img.protocol != CCL_PROTO_SIMPLE) return refuse("generated kernels cover the flag protocol only");
    if ((int)img.tb_segs.size() != img.ntb) return refuse("plan has no segment structure");
    const bool seq = img.engine == CCL_ENGINE_SEQUENTIAL;
    const int m = img.m;
    const int es = img.esize;
    const long long ve = 16 / es;
    const long long slot_elems = img.slot_bytes / es;
    const long long S = img.S;

    // ---- replay every threadblock program and derive the per-instruction forms
    std::vector<std::vector<InstrForm>> forms(img.ntb);
    size_t total_blocks = 0;
    for (int b = 0; b < img.ntb; ++b) {
        const int k0 = img.tb_begin[b], k1 = img.tb_begin[b + 1];
        std::map<int, std::vector<int>> steps_of;   // ci -> step indices
        std::map<int, int> pos_of;                  // ci -> position in its segment
        std::map<int, int> seg_of;
        std::vector<long long> seg_base;            // first step of every segment
        {
            int k = k0;
            for (size_t g = 0; g < img.tb_segs[b].size(); ++g) {
                const SegInfo& seg = img.tb_segs[b][g];
                seg_base.push_back(k);
                for (size_t p = 0; p < seg.cis.size(); ++p) {
                    pos_of[seg.cis[p]] = (int)p;
                    seg_of[seg.cis[p]] = (int)g;
                }
                for (int w0 = 0; w0 < m; w0 += seg.window) {
                    const int w1 = std::min(m, w0 + seg.window);
                    for (int ci : seg.cis)
                        for (int mb = w0; mb < w1; ++mb, ++k) {
                            if (k >= k1 || img.steps[k].instr != ci || img.steps[k].mb != mb)
                                return refuse("threadblock " + std::to_string(b) + " does not follow its segments");
                            steps_of[ci].push_back(k);
                        }
                }
            }
            if (k != k1) return refuse("threadblock " + std::to_string(b) + " has steps outside its segments");
        }
        // running sequence numbers per link, pieces and slot counts
        std::map<int, long long> qin, qout;
        for (int k = k0; k < k1; ++k) {
            const DStep& st = img.steps[k];
            const DInstr& D = img.instrs[st.instr];
            long long off = 0, len = 0;
            {
                const long long V = D.nelem / ve;
                off = (V * st.mb / m) * ve;
                len = (st.mb == m - 1 ? D.nelem : (V * (st.mb + 1) / m) * ve) - off;
            }
            const bool linked = D.link_in >= 0 || D.link_out >= 0;
            const long long ns = linked ? std::max<long long>(1, (len + slot_elems - 1) / slot_elems) : 0;
            if (st.elem_off != off || st.nelem != len || st.nslots != ns)
                return refuse("a piece does not follow the split formula");
            if (st.flags & STEP_NOPOST) return refuse("a step carries the test hook that drops its signals");
            if (D.link_in >= 0) {
                if (st.seq_in != qin[D.link_in]) return refuse("a link is received in another order than sent");
                qin[D.link_in] += ns;
            }
            if (D.link_out >= 0) {
                if (st.seq_out != qout[D.link_out]) return refuse("sequence numbers do not follow the sender");
                qout[D.link_out] += ns;
            }
        }
        for (auto& e : steps_of) {
            const int ci = e.first;
            const std::vector<int>& ks = e.second;
            InstrForm f;
            f.ci = ci;
            f.signal = img.steps[ks[0]].signal;
            f.flags = img.steps[ks[0]].flags;
            // dependency counters: present at every piece -> exact, only at
            // piece 0 -> whole
            std::map<int, int> seen;
            for (int k : ks)
                for (auto& d : step_deps(img, img.steps[k])) seen[d.first]++;
            for (auto& c : seen) {
                if (c.second == (int)ks.size() && (int)ks.size() > 0) f.deps.exact.push_back(c.first);
                else if (c.second == 1) f.deps.whole.push_back(c.first);
                else return refuse("irregular dependency counters");
            }
            // counters both exact and at piece 0 with value m
            for (int c : f.deps.exact) {
                const DepSet s0 = step_deps(img, img.steps[ks[0]]);
                for (auto& d : s0)
                    if (d.first == c && d.second == m && m > 1) f.deps.whole.push_back(c);
            }
            // drain (the pipelined engine's issuer waits for an earlier step
            // of its own threadblock): the first of the forms that names the
            // planner's step at every piece
            const DStep& s0 = img.steps[ks[0]];
            if (!seq && s0.drain >= 0) {
                InstrForm cand[3] = {f, f, f};
                cand[0].drain_kind = 2;
                cand[0].drain_const = s0.drain;
                cand[1].drain_kind = 3;
                cand[1].drain_dk = ks[0] - s0.drain;
                cand[2].drain_kind = 4;   // the producer of the first piece, same micro-batch
                const int pc = img.steps[s0.drain].instr;
                if (seg_of.count(pc)) {
                    const SegInfo& ps = img.tb_segs[b][seg_of[pc]];
                    cand[2].p_base = seg_base[seg_of[pc]];
                    cand[2].p_n = (int)ps.cis.size();
                    cand[2].p_w = ps.window;
                    cand[2].p_pos = pos_of[pc];
                }
                f.drain_kind = -1;
                for (const InstrForm& c : cand) {
                    bool ok = true;
                    for (int k : ks) ok = ok && drain_of(c, k, img.steps[k].mb, m) == img.steps[k].drain;
                    if (ok) {
                        f = c;
                        break;
                    }
                }
                if (f.drain_kind < 0) {
                    std::string d;
                    for (int k : ks)
                        d += " " + std::to_string(k) + "(mb " + std::to_string(img.steps[k].mb) + ")->" +
                             std::to_string(img.steps[k].drain);
                    return refuse("irregular drains of threadblock " + std::to_string(b) + " instruction " +
                                  std::to_string(ci) + ":" + d.substr(0, 600));
                }
            }
            // verify deps, signal, flags and drain at every piece
            for (int k : ks) {
                const DStep& st = img.steps[k];
                if (st.signal != f.signal || st.flags != f.flags) return refuse("irregular signal counters or hints");
                if (form_deps(f.deps, st.mb, m) != step_deps(img, st)) return refuse("irregular dependency counters");
                if (!seq && drain_of(f, k, st.mb, m) != st.drain) return refuse("irregular drains");
            }
            forms[b].push_back(f);
        }
        total_blocks += steps_of.size();
    }

    // ---- emit: the constants of every instruction of every threadblock as
    // one table of the generated module (compiled in, read-only), then per
    // threadblock its segments' window loops calling the shared block
    // function on its instructions' entries
    std::string o;
    o += "// Kernel generated for one plan (see ccl_codegen.cpp).\n";
    o += "#include \"ccl_core.cuh\"\nnamespace ccl {\n";
    (void)total_blocks;
    const int U = build <= 512 ? 8 : 4;
    const std::string geom = std::to_string(m) + ", " + lit(ve) + ", " + lit(slot_elems) + ", " + std::to_string(S);
    // table entries in threadblock and segment order, so that every segment's
    // instructions are one contiguous range
    std::string table, dep_list;
    int nentries = 0, ndeps = 0;
    std::vector<std::vector<int>> seg_first(img.ntb);
    std::vector<int> nq(img.ntb, 0);
    std::vector<int> prog_first(img.ntb + 1, 0), dep_first_of(img.ntb + 1, 0);   // each program's entries
    for (int b = 0; b < img.ntb; ++b) {
        prog_first[b] = nentries;
        dep_first_of[b] = ndeps;
        std::map<int, const InstrForm*> form_of;
        for (const InstrForm& f : forms[b]) form_of[f.ci] = &f;
        std::map<int, int> qin_slot, qout_slot;   // link -> this threadblock's counter
        for (const SegInfo& seg : img.tb_segs[b]) {
            seg_first[b].push_back(nentries);
            for (int ci : seg.cis) {
                const InstrForm& f = *form_of.at(ci);
                const DInstr& D = img.instrs[ci];
                int qi = -1, qo = -1;
                if (D.link_in >= 0) {
                    if (!qin_slot.count(D.link_in)) qin_slot[D.link_in] = nq[b]++;
                    qi = qin_slot[D.link_in];
                }
                if (D.link_out >= 0) {
                    if (!qout_slot.count(D.link_out)) qout_slot[D.link_out] = nq[b]++;
                    qo = qout_slot[D.link_out];
                }
                auto link = [&](int L) {
                    if (L < 0) return std::string("{0, 0, 0, 0, 0, 0}");
                    const DLink& K = img.links[L];
                    return "{" + lit(K.slot_base) + ", " + lit(K.total) + ", " + std::to_string(K.flag_base) + ", " +
                           std::to_string(K.src_rank) + ", " + std::to_string(K.dst_rank) + ", " +
                           std::to_string(K.total_mod) + "}";
                };
                std::set<int> whole(f.deps.whole.begin(), f.deps.whole.end());
                std::vector<std::pair<int, int>> deps;   // counter, bit 0 exact | bit 1 whole
                for (int c : f.deps.exact) deps.push_back({c, 1 | (whole.count(c) ? 2 : 0)});
                std::set<int> exact(f.deps.exact.begin(), f.deps.exact.end());
                for (int c : f.deps.whole)
                    if (!exact.count(c)) deps.push_back({c, 2});
                const int dep_first = ndeps;
                for (auto& d : deps) {
                    dep_list += (ndeps % 8 ? " {" : (ndeps ? "\n    {" : "    {")) + std::to_string(d.first) + ", " +
                                std::to_string(d.second) + "},";
                    ++ndeps;
                }
                // DRec: kind dtype link_in link_out src_buf src_rank loc_buf loc_rank dst_buf dst_rank
                // nslots dep_begin dep_count signal mb flags src_off loc_off dst_off nelem seq_in
                // seq_out drain seq_in_mod seq_out_mod link_loc x_buf x_rank x_off (nelem: the whole
                // channel range)
                table += "    {{" + std::to_string(D.kind) + ", " + std::to_string(D.dtype) + ", " +
                         std::to_string(D.link_in) + ", " + std::to_string(D.link_out) + ", " + std::to_string(D.src_buf) +
                         ", " + std::to_string(D.src_rank) + ", " + std::to_string(D.loc_buf) + ", " +
                         std::to_string(D.loc_rank) + ", " + std::to_string(D.dst_buf) + ", " + std::to_string(D.dst_rank) +
                         ", 0, 0, 0, " + std::to_string(f.signal) + ", 0, " + std::to_string(f.flags) + ", " +
                         lit(D.src_off) + ", " + lit(D.loc_off) + ", " + lit(D.dst_off) + ", " + lit(D.nelem) +
                         ", 0, 0, -1, 0, 0, 0, " + std::to_string(D.x_buf) + ", " + std::to_string(D.x_rank) + ", " +
                         lit(D.x_buf >= 0 ? D.x_off : 0) + "}, " + link(D.link_in) + ", " + link(D.link_out) + ", " +
                         std::to_string(dep_first) + ", " + std::to_string(deps.size()) + ", " +
                         std::to_string(seq ? 0 : f.drain_kind) + ", " + std::to_string(f.drain_dk) + ", " +
                         std::to_string(f.drain_const) + ", " + lit(f.p_base) + ", " + std::to_string(f.p_n) + ", " +
                         std::to_string(f.p_w) + ", " + std::to_string(f.p_pos) + ", " + std::to_string(qi) + ", " +
                         std::to_string(qo) + "},\n";
                ++nentries;
            }
        }
    }
    prog_first[img.ntb] = nentries;
    dep_first_of[img.ntb] = ndeps;
    // Each program copies its own entries (and their dependency lists, with
    // dep_first rebased) into shared memory at start when they fit: reads of
    // the table from global memory would go to L2 at every piece (the waits'
    // acquire fences drop L1 lines).  kTabMax entries of at most 256 bytes.
    int max_n = 0, max_d = 0;
    for (int b = 0; b < img.ntb; ++b) {
        max_n = std::max(max_n, prog_first[b + 1] - prog_first[b]);
        max_d = std::max(max_d, dep_first_of[b + 1] - dep_first_of[b]);
    }
    const bool shared_tab = max_n > 0 && max_n <= 96 && max_n * 256 + max_d * 8 <= 28 * 1024;
    auto ints = [](const std::vector<int>& v) {
        std::string r;
        for (size_t i = 0; i < v.size(); ++i) r += (i ? ", " : "") + std::to_string(v[i]);
        return r;
    };
    o += "static __device__ const GenInstr kGen[" + std::to_string(std::max(1, nentries)) + "] = {\n" +
         (nentries ? table : std::string("    {}\n")) + "};\n";
    o += "static __device__ const int2 kGenDep[" + std::to_string(std::max(1, ndeps)) + "] = {\n" +
         (ndeps ? dep_list : std::string("    {0, 0}")) + "\n};\n";
    o += "static __device__ const int kProgFirst[" + std::to_string(img.ntb + 1) + "] = {" + ints(prog_first) + "};\n";
    o += "static __device__ const int kDepFirst[" + std::to_string(img.ntb + 1) + "] = {" + ints(dep_first_of) + "};\n";
    for (int b = 0; b < img.ntb; ++b) {
        // tab: the program's entries (tab[j - first of the program]); dep:
        // the dependency list its entries index
        if (seq)
            o += "static __device__ __noinline__ void gtb" + std::to_string(b) +
                 "(const KParams& P, int* go, GenStep* gs, const GenInstr* tab, const int2* dep)\n{\n";
        else
            o += "static __device__ __noinline__ void gtb" + std::to_string(b) +
                 "(const KParams& P, CtlShared* sh, const GenInstr* tab, const int2* dep)\n{\n";
        o += "    const unsigned exec_mod = (unsigned)(P.exec % P.S);\n";
        if (!seq) o += "    int head = 0;\n";
        o += "    int si = " + std::to_string(img.tb_begin[b]) + ";\n";
        o += "    long long q[" + std::to_string(std::max(1, nq[b])) + "] = {};\n";
        for (size_t g = 0; g < img.tb_segs[b].size(); ++g) {
            const SegInfo& seg = img.tb_segs[b][g];
            const int first = seg_first[b][g], n = (int)seg.cis.size();
            // loops stay loops: one call site per segment
            o += "#pragma unroll 1\n    for (int w0 = 0; w0 < " + std::to_string(m) + "; w0 += " +
                 std::to_string(seg.window) + ") {\n";
            o += "        const int w1 = w0 + " + std::to_string(seg.window) + " < " + std::to_string(m) + " ? w0 + " +
                 std::to_string(seg.window) + " : " + std::to_string(m) + ";\n";
            o += "#pragma unroll 1\n        for (int j = " + std::to_string(first) + "; j < " + std::to_string(first + n) +
                 "; ++j)\n";
            const std::string entry = "tab[j - " + std::to_string(prog_first[b]) + "]";
            if (seq)
                o += "            if (!gen_seq_block<" + std::to_string(U) + ">(P, go, gs, " + entry + ", dep, w0, w1, " +
                     geom + ", si, q, exec_mod)) return;\n";
            else
                o += "            if (!gen_issue_block(P, sh, " + entry + ", dep, w0, w1, " + geom +
                     ", si, head, q, exec_mod)) return;\n";
            o += "    }\n";
        }
        if (!seq) o += "    publish_cmd(sh, head, 1, 4 * P.timeout_ns);\n";
        o += "    (void)exec_mod;\n}\n";
    }
    o += "}  // namespace ccl\n\n";
    const std::string maxt = std::to_string(build <= 512 ? 512 : 1024);
    o += "extern \"C\" __global__ void __launch_bounds__(" + maxt +
         ", 1) ccl_gen_kernel(const __grid_constant__ ccl::KParams P)\n{\n";
    const std::string prog = seq ? "(P.cluster > 1 ? blockIdx.x / P.cluster : blockIdx.x)" : "blockIdx.x";
    std::string sw = "switch (" + prog + ") {\n";
    for (int b = 0; b < img.ntb; ++b)
        sw += "    case " + std::to_string(b) + ": ccl::gtb" + std::to_string(b) +
              (seq ? "(P, &go_flag, &gstep, gtab, gdep)" : "(P, &sh, gtab, gdep)") + "; break;\n";
    // the program's table: a copy in shared memory, or the module's arrays
    std::string tabinit;
    if (shared_tab) {
        tabinit += "    __shared__ __align__(16) ccl::GenInstr gtab_s[" + std::to_string(max_n) + "];\n";
        tabinit += "    __shared__ int2 gdep_s[" + std::to_string(std::max(1, max_d)) + "];\n";
        tabinit += "    {\n        const int pg = " + prog + ";\n";
        tabinit += "        const int e0 = ccl::kProgFirst[pg], n = ccl::kProgFirst[pg + 1] - e0;\n";
        tabinit += "        const int d0 = ccl::kDepFirst[pg], nd = ccl::kDepFirst[pg + 1] - d0;\n";
        tabinit += "        if ((int)threadIdx.x < n) {\n            ccl::GenInstr g = ccl::kGen[e0 + threadIdx.x];\n";
        tabinit += "            g.dep_first -= d0;\n            gtab_s[threadIdx.x] = g;\n        }\n";
        tabinit += "        for (int i = threadIdx.x; i < nd; i += blockDim.x) gdep_s[i] = ccl::kGenDep[d0 + i];\n    }\n";
        tabinit += "    const ccl::GenInstr* gtab = gtab_s;\n    const int2* gdep = gdep_s;\n";
    } else {
        tabinit += "    const ccl::GenInstr* gtab = ccl::kGen + ccl::kProgFirst[" + prog + "];\n";
        tabinit += "    const int2* gdep = ccl::kGenDep;\n";
    }
    sw += "    default: break;\n    }\n";
    o += tabinit;
    if (seq) {
        o += "    __shared__ int go_flag;\n    __shared__ __align__(16) ccl::GenStep gstep;\n";
        o += "    // every CTA of the cluster has started; the table is in place\n";
        o += "    ccl::group_sync(P);\n    " + sw;
    } else {
        o += "    __shared__ __align__(16) ccl::CtlShared sh;\n";
        o += "    extern __shared__ __align__(128) unsigned char stages[];\n";
        o += "    ccl::ctl_init(P, &sh);   // its barrier also publishes the table\n";
        o += "    const int warp = threadIdx.x >> 5;\n";
        o += "    if (warp < 3) {\n        if ((threadIdx.x & 31) == 0) {\n            if (warp == 0) {\n";
        o += "    " + sw;
        o += "            } else if (warp == 1) {\n                ccl::releaser(P, &sh);\n            } else {\n"
             "                ccl::tma_thread(P, &sh, stages);\n            }\n        }\n        return;\n    }\n";
        o += "    ccl::data_warps<false, " + maxt + ">(P, &sh);\n";
    }
    o += "}\n";
    return o;
}

}  // namespace ccl
