// Internal structures shared by the host compiler, the planner and the
// runtime.  Not part of the C ABI.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "../../include/ccl.h"

namespace ccl {

// ---------------------------------------------------------------- errors
void set_error(const std::string& msg);
ccl_status_t fail(ccl_status_t st, const std::string& msg);

// ---------------------------------------------------------------- ranges
struct Range {
    int32_t rank = -1;
    int32_t buf = -1;
    int64_t off = 0;   // chunks
    int64_t cnt = 0;   // chunks
    bool valid() const { return rank >= 0; }
    bool same(const Range& o) const {
        return rank == o.rank && buf == o.buf && off == o.off && cnt == o.cnt;
    }
    bool overlaps(const Range& o) const {
        return rank >= 0 && o.rank >= 0 && rank == o.rank && buf == o.buf && off < o.off + o.cnt &&
               o.off < off + cnt;
    }
};

// ------------------------------------------------------ fused instruction
// A rank-level instruction after lowering and fusion (before the channel /
// micro-batch split).  Reads `src` and/or `loc`, receives `xfer_in`,
// writes `dst`, sends `xfer_out`.
struct Instr {
    int kind = CCL_I_COPY;   // ccl_instr_kind_t
    int rank = -1;
    Range src, loc, dst;
    Range x;                 // second destination of a folded receive (plans only)
    int64_t count = 0;       // chunks
    int xfer_in = -1, xfer_out = -1;
    int position = 0;        // program position (order on its rank)
};

struct Xfer {
    int src_rank = -1, dst_rank = -1;
    int send_instr = -1, recv_instr = -1;
    int64_t count = 0;
    int chunk_id = 0;        // data identity used by the HPDS priority
    int op_index = 0;        // operation of the source program
};

// dependency of instruction `to` on instruction `from` (same rank, buffer
// hazard).  exact: the hazard is between identical ranges, so micro-batch j
// of `to` only needs micro-batch j of `from`.
struct Dep {
    int from, to;
    bool exact;
};

}  // namespace ccl

struct ccl_schedule {
    int32_t nranks = 0;
    int32_t nchunks[3] = {0, 0, 0};
    int32_t builtin = -1;
    int32_t group_size = 0;
    int32_t fuse = CCL_FUSE_FULL;     // fusion mode the instructions were compiled with
    std::vector<ccl_op_t> ops;
    std::vector<ccl::Instr> instrs;   // sorted by (rank, position)
    std::vector<ccl::Xfer> xfers;
    std::vector<ccl::Dep> deps;       // same-rank buffer hazards between instructions
};

namespace ccl {

int64_t kind_bytes_factor(int kind);   // bytes moved per element byte
bool kind_reads_slot(int kind);
bool kind_writes_slot(int kind);
bool kind_is_reduce(int kind);
// fuse: CCL_FUSE_NONE, CCL_FUSE_FULL or CCL_FUSE_NOCHAIN
ccl_status_t compile_program(const ccl_op_t* ops, int nops, int nranks, const int32_t nchunks[3],
                             int fuse, ccl_schedule* s);
int fuse_mode(uint32_t flags);
ccl_status_t builtin_program(int kind, int nranks, int G, uint32_t flags,
                             std::vector<ccl_op_t>* ops, int32_t nchunks[3]);
// uneven AllToAll: counts[s * R + d] chunks from s to d
ccl_status_t alltoallv_program(int R, const int32_t* counts, std::vector<ccl_op_t>* ops, int32_t nchunks[3]);

}  // namespace ccl
