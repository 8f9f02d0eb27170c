// Persistence of compiled schedules and of per-size tuning tables as JSON
// files, and the lookup of a tuned configuration by message size.
//
// A schedule file holds the source program (ops, chunk counts, fusion mode,
// built-in kind) and a digest of the fused instruction list; reading it
// compiles the program again and refuses a file whose digest no longer
// matches (the compiler changed since it was written).  A tuning table holds,
// per message size, the configuration the tuner chose (AutoCCL report,
// research method 1-2: parameters tuned per message size) with its timings.
//
// The JSON reader accepts the subset these writers produce: objects, arrays,
// numbers, strings without escapes other than \" and \\, true/false/null.
#include <cctype>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <memory>
#include <string>
#include <vector>

#include "ccl_internal.h"

namespace ccl {
namespace {

// ------------------------------------------------------------ JSON values
struct JVal {
    enum T { NUL, BOOL, NUM, STR, ARR, OBJ } t = NUL;
    double num = 0;
    std::string str;
    std::vector<JVal> arr;
    std::map<std::string, JVal> obj;
    const JVal* get(const std::string& k) const
    {
        auto it = obj.find(k);
        return t == OBJ && it != obj.end() ? &it->second : nullptr;
    }
};

class Parser {
public:
    explicit Parser(const std::string& s) : s_(s) {}
    bool parse(JVal* v)
    {
        if (!value(v)) return false;
        ws();
        return i_ == s_.size();
    }
    std::string error;

private:
    const std::string& s_;
    size_t i_ = 0;
    void ws()
    {
        while (i_ < s_.size() && std::isspace((unsigned char)s_[i_])) ++i_;
    }
    bool bad(const char* what)
    {
        error = std::string(what) + " at offset " + std::to_string(i_);
        return false;
    }
    bool value(JVal* v)
    {
        ws();
        if (i_ >= s_.size()) return bad("unexpected end");
        char c = s_[i_];
        if (c == '{') return object(v);
        if (c == '[') return array(v);
        if (c == '"') { v->t = JVal::STR; return string(&v->str); }
        if (s_.compare(i_, 4, "true") == 0) { v->t = JVal::BOOL; v->num = 1; i_ += 4; return true; }
        if (s_.compare(i_, 5, "false") == 0) { v->t = JVal::BOOL; v->num = 0; i_ += 5; return true; }
        if (s_.compare(i_, 4, "null") == 0) { v->t = JVal::NUL; i_ += 4; return true; }
        const char* b = s_.c_str() + i_;
        char* e = nullptr;
        v->num = std::strtod(b, &e);
        if (e == b) return bad("bad value");
        v->t = JVal::NUM;
        i_ += (size_t)(e - b);
        return true;
    }
    bool string(std::string* out)
    {
        ++i_;   // opening quote
        out->clear();
        while (i_ < s_.size() && s_[i_] != '"') {
            if (s_[i_] == '\\' && i_ + 1 < s_.size()) ++i_;
            out->push_back(s_[i_++]);
        }
        if (i_ >= s_.size()) return bad("unterminated string");
        ++i_;
        return true;
    }
    bool array(JVal* v)
    {
        v->t = JVal::ARR;
        ++i_;
        ws();
        if (i_ < s_.size() && s_[i_] == ']') { ++i_; return true; }
        while (true) {
            v->arr.emplace_back();
            if (!value(&v->arr.back())) return false;
            ws();
            if (i_ < s_.size() && s_[i_] == ',') { ++i_; continue; }
            if (i_ < s_.size() && s_[i_] == ']') { ++i_; return true; }
            return bad("expected , or ]");
        }
    }
    bool object(JVal* v)
    {
        v->t = JVal::OBJ;
        ++i_;
        ws();
        if (i_ < s_.size() && s_[i_] == '}') { ++i_; return true; }
        while (true) {
            ws();
            if (i_ >= s_.size() || s_[i_] != '"') return bad("expected a key");
            std::string k;
            if (!string(&k)) return false;
            ws();
            if (i_ >= s_.size() || s_[i_] != ':') return bad("expected :");
            ++i_;
            if (!value(&v->obj[k])) return false;
            ws();
            if (i_ < s_.size() && s_[i_] == ',') { ++i_; continue; }
            if (i_ < s_.size() && s_[i_] == '}') { ++i_; return true; }
            return bad("expected , or }");
        }
    }
};

ccl_status_t read_file(const char* path, std::string* out)
{
    if (!path) return fail(CCL_ERR_INVALID_ARG, "null path");
    std::FILE* f = std::fopen(path, "rb");
    if (!f) return fail(CCL_ERR_INVALID_ARG, std::string("cannot open ") + path);
    char buf[65536];
    size_t n;
    out->clear();
    while ((n = std::fread(buf, 1, sizeof(buf), f)) > 0) out->append(buf, n);
    std::fclose(f);
    return CCL_OK;
}

ccl_status_t write_file(const char* path, const std::string& text)
{
    if (!path) return fail(CCL_ERR_INVALID_ARG, "null path");
    std::string tmp = std::string(path) + ".tmp";
    std::FILE* f = std::fopen(tmp.c_str(), "wb");
    if (!f) return fail(CCL_ERR_INVALID_ARG, std::string("cannot write ") + tmp);
    bool ok = std::fwrite(text.data(), 1, text.size(), f) == text.size();
    ok = std::fclose(f) == 0 && ok;
    if (!ok || std::rename(tmp.c_str(), path) != 0) {
        std::remove(tmp.c_str());
        return fail(CCL_ERR_INVALID_ARG, std::string("cannot write ") + path);
    }
    return CCL_OK;
}

ccl_status_t parse_text(const std::string& text, JVal* root)
{
    Parser p(text);
    if (!p.parse(root) || root->t != JVal::OBJ) return fail(CCL_ERR_INVALID_ARG, "malformed JSON: " + p.error);
    return CCL_OK;
}

bool num(const JVal* v, double* out)
{
    if (!v || (v->t != JVal::NUM && v->t != JVal::BOOL)) return false;
    *out = v->num;
    return true;
}

// FNV-1a over the fields of every fused instruction
uint64_t instr_digest(const ccl_schedule& s)
{
    uint64_t h = 1469598103934665603ull;
    auto mix = [&](int64_t x) {
        for (int b = 0; b < 8; ++b) {
            h ^= (uint64_t)((x >> (8 * b)) & 0xff);
            h *= 1099511628211ull;
        }
    };
    for (const Instr& I : s.instrs) {
        mix(I.kind); mix(I.rank); mix(I.count); mix(I.xfer_in); mix(I.xfer_out); mix(I.position);
        for (const Range* r : {&I.src, &I.loc, &I.dst}) { mix(r->rank); mix(r->buf); mix(r->off); mix(r->cnt); }
    }
    return h;
}

// the fields of ccl_plan_opts_t by name (the file names them, so a reader
// does not depend on the field order)
struct OptField {
    const char* name;
    int64_t (*get)(const ccl_plan_opts_t&);
    void (*set)(ccl_plan_opts_t&, int64_t);
};
#define OPT_FIELD(f) \
    OptField{#f, [](const ccl_plan_opts_t& o) { return (int64_t)o.f; }, [](ccl_plan_opts_t& o, int64_t v) { o.f = (decltype(o.f))v; }}
const OptField kOptFields[] = {
    OPT_FIELD(channels), OPT_FIELD(nthreads), OPT_FIELD(slot_bytes), OPT_FIELD(fifo_slots),
    OPT_FIELD(microbatches), OPT_FIELD(scheduler), OPT_FIELD(tb_alloc), OPT_FIELD(mb_order),
    OPT_FIELD(timeout_ms), OPT_FIELD(instrument), OPT_FIELD(tile_bytes), OPT_FIELD(bulk),
    OPT_FIELD(link_mode), OPT_FIELD(channel_scaling), OPT_FIELD(mb_window), OPT_FIELD(protocol),
    OPT_FIELD(tb_budget), OPT_FIELD(engine), OPT_FIELD(codegen), OPT_FIELD(cluster), OPT_FIELD(fold)};
#undef OPT_FIELD

std::string fmt_double(double x)
{
    char b[64];
    std::snprintf(b, sizeof(b), "%.17g", std::isfinite(x) ? x : 0.0);
    return b;
}

}  // namespace
}  // namespace ccl

extern "C" {

ccl_status_t ccl_schedule_write_json(ccl_schedule_t s, const char* path)
{
    using namespace ccl;
    if (!s) return fail(CCL_ERR_INVALID_ARG, "null schedule");
    std::string t = "{\n  \"format\": \"ccl-schedule-1\",\n";
    t += "  \"nranks\": " + std::to_string(s->nranks) + ",\n";
    t += "  \"nchunks\": [" + std::to_string(s->nchunks[0]) + ", " + std::to_string(s->nchunks[1]) + ", " +
         std::to_string(s->nchunks[2]) + "],\n";
    t += "  \"fuse\": " + std::to_string(s->fuse) + ",\n";
    t += "  \"builtin\": " + std::to_string(s->builtin) + ",\n";
    t += "  \"group_size\": " + std::to_string(s->group_size) + ",\n";
    t += "  \"ninstr\": " + std::to_string(s->instrs.size()) + ",\n";
    t += "  \"instr_digest\": \"" + std::to_string(instr_digest(*s)) + "\",\n";
    t += "  \"ops\": [";
    for (size_t i = 0; i < s->ops.size(); ++i) {
        const ccl_op_t& o = s->ops[i];
        t += std::string(i ? ",\n    " : "\n    ") + "[" + std::to_string(o.op) + ", " + std::to_string(o.src_rank) +
             ", " + std::to_string(o.src_buf) + ", " + std::to_string(o.src_off) + ", " + std::to_string(o.dst_rank) +
             ", " + std::to_string(o.dst_buf) + ", " + std::to_string(o.dst_off) + ", " + std::to_string(o.count) +
             "]";
    }
    t += "\n  ]\n}\n";
    return write_file(path, t);
}

ccl_status_t ccl_schedule_read_json(const char* path, ccl_schedule_t* out)
{
    using namespace ccl;
    if (!out) return fail(CCL_ERR_INVALID_ARG, "null argument");
    std::string text;
    ccl_status_t st = read_file(path, &text);
    if (st != CCL_OK) return st;
    JVal root;
    if ((st = parse_text(text, &root)) != CCL_OK) return st;
    const JVal* fmt = root.get("format");
    if (!fmt || fmt->t != JVal::STR || fmt->str != "ccl-schedule-1")
        return fail(CCL_ERR_INVALID_ARG, "not a ccl-schedule-1 file");
    double nranks, fuse, builtin, group;
    const JVal* nch = root.get("nchunks");
    const JVal* ops = root.get("ops");
    const JVal* dig = root.get("instr_digest");
    if (!num(root.get("nranks"), &nranks) || !num(root.get("fuse"), &fuse) || !num(root.get("builtin"), &builtin) ||
        !num(root.get("group_size"), &group) || !nch || nch->t != JVal::ARR || nch->arr.size() != 3 || !ops ||
        ops->t != JVal::ARR || !dig || dig->t != JVal::STR)
        return fail(CCL_ERR_INVALID_ARG, "schedule file lacks a field");
    int32_t nc[3];
    for (int b = 0; b < 3; ++b) {
        double x;
        if (!num(&nch->arr[b], &x)) return fail(CCL_ERR_INVALID_ARG, "bad chunk count");
        nc[b] = (int32_t)x;
    }
    std::vector<ccl_op_t> prog;
    for (const JVal& row : ops->arr) {
        if (row.t != JVal::ARR || row.arr.size() != 8) return fail(CCL_ERR_INVALID_ARG, "bad operation row");
        int32_t f[8];
        for (int k = 0; k < 8; ++k) {
            double x;
            if (!num(&row.arr[k], &x)) return fail(CCL_ERR_INVALID_ARG, "bad operation field");
            f[k] = (int32_t)x;
        }
        prog.push_back(ccl_op_t{f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]});
    }
    std::unique_ptr<ccl_schedule> s(new ccl_schedule());
    st = compile_program(prog.data(), (int)prog.size(), (int)nranks, nc, (int)fuse, s.get());
    if (st != CCL_OK) return st;
    s->builtin = (int32_t)builtin;
    s->group_size = (int32_t)group;
    if (std::to_string(instr_digest(*s)) != dig->str)
        return fail(CCL_ERR_INVALID_ARG, "the program compiles to other instructions than when it was written");
    *out = s.release();
    return CCL_OK;
}

ccl_status_t ccl_tune_table_write_json(const ccl_tune_row_t* rows, int32_t n, int32_t dtype, const char* note,
                                       const char* path)
{
    using namespace ccl;
    if (n < 0 || (n > 0 && !rows)) return fail(CCL_ERR_INVALID_ARG, "bad rows");
    std::string t = "{\n  \"format\": \"ccl-tune-table-1\",\n  \"dtype\": " + std::to_string(dtype) + ",\n";
    std::string nt = note ? note : "";
    for (char& c : nt)
        if (c == '"' || c == '\\' || c == '\n') c = ' ';
    t += "  \"note\": \"" + nt + "\",\n  \"rows\": [";
    for (int i = 0; i < n; ++i) {
        const ccl_tune_row_t& r = rows[i];
        t += std::string(i ? ",\n    " : "\n    ") + "{\"chunk_elems\": " + std::to_string(r.chunk_elems) +
             ", \"probes\": " + std::to_string(r.report.probes) + ", \"best_us\": " + fmt_double(r.report.best_us) +
             ", \"best_gbs\": " + fmt_double(r.report.best_gbs) + ", \"default_us\": " +
             fmt_double(r.report.default_us) + ", \"opts\": {";
        bool first = true;
        for (const OptField& f : kOptFields) {
            t += std::string(first ? "" : ", ") + "\"" + f.name + "\": " + std::to_string(f.get(r.best));
            first = false;
        }
        t += "}}";
    }
    t += "\n  ]\n}\n";
    return write_file(path, t);
}

ccl_status_t ccl_tune_table_read_json(const char* path, ccl_tune_row_t* rows, int32_t cap, int32_t* n,
                                      int32_t* dtype)
{
    using namespace ccl;
    if (!n) return fail(CCL_ERR_INVALID_ARG, "null argument");
    std::string text;
    ccl_status_t st = read_file(path, &text);
    if (st != CCL_OK) return st;
    JVal root;
    if ((st = parse_text(text, &root)) != CCL_OK) return st;
    const JVal* fmt = root.get("format");
    const JVal* rs = root.get("rows");
    double dt;
    if (!fmt || fmt->t != JVal::STR || fmt->str != "ccl-tune-table-1" || !rs || rs->t != JVal::ARR ||
        !num(root.get("dtype"), &dt))
        return fail(CCL_ERR_INVALID_ARG, "not a ccl-tune-table-1 file");
    *n = (int32_t)rs->arr.size();
    if (dtype) *dtype = (int32_t)dt;
    if (!rows) return CCL_OK;
    if (cap < *n) return fail(CCL_ERR_INVALID_ARG, "capacity too small");
    for (int i = 0; i < *n; ++i) {
        const JVal& r = rs->arr[i];
        ccl_tune_row_t& o = rows[i];
        std::memset(&o, 0, sizeof(o));
        ccl_plan_opts_default(&o.best);
        double ce, probes = 0;
        if (!num(r.get("chunk_elems"), &ce)) return fail(CCL_ERR_INVALID_ARG, "row without chunk_elems");
        o.chunk_elems = (int64_t)ce;
        num(r.get("probes"), &probes);
        o.report.probes = (int32_t)probes;
        num(r.get("best_us"), &o.report.best_us);
        num(r.get("best_gbs"), &o.report.best_gbs);
        num(r.get("default_us"), &o.report.default_us);
        const JVal* opts = r.get("opts");
        if (!opts || opts->t != JVal::OBJ) return fail(CCL_ERR_INVALID_ARG, "row without opts");
        for (const OptField& f : kOptFields) {
            double x;
            if (num(opts->get(f.name), &x)) f.set(o.best, (int64_t)x);
        }
    }
    return CCL_OK;
}

ccl_status_t ccl_tune_table_lookup(const ccl_tune_row_t* rows, int32_t n, int64_t chunk_elems, ccl_plan_opts_t* out)
{
    using namespace ccl;
    if (!rows || n <= 0 || !out || chunk_elems <= 0) return fail(CCL_ERR_INVALID_ARG, "bad arguments");
    int best = -1;
    double bd = 0;
    for (int i = 0; i < n; ++i) {
        if (rows[i].chunk_elems <= 0) continue;
        const double d = std::fabs(std::log((double)rows[i].chunk_elems / (double)chunk_elems));
        if (best < 0 || d < bd - 1e-12) { best = i; bd = d; }
    }
    if (best < 0) return fail(CCL_ERR_INVALID_ARG, "table has no usable row");
    *out = rows[best].best;
    return CCL_OK;
}

}  // extern "C"
