// Host-side plan image: everything the executor kernel reads, built by the
// planner from a compiled schedule and the execution parameters.
#pragma once

#include <cstdint>
#include <vector>

#include "ccl_internal.h"
#include "ccl_layout.h"

namespace ccl {

// operand buffer classes (select cache hints in the kernel)
enum : int32_t { OPB_NONE = -1 };

// One channel instruction.  Offsets are element offsets of the channel
// range inside the rank's buffer; a missing operand has buf = -1.
struct DInstr {
    int32_t kind;
    int32_t dtype;
    int32_t link_in, link_out;
    int32_t src_rank, src_buf;
    int32_t loc_rank, loc_buf;
    int32_t dst_rank, dst_buf;
    int32_t x_rank, x_buf;          // second destination (buf -1: none)
    int64_t src_off, loc_off, dst_off;
    int64_t nelem;
    int64_t x_off;
};
static_assert(sizeof(DInstr) == 88, "DInstr layout");

// One (channel instruction, micro-batch) step of a threadblock program.
struct DStep {
    int32_t instr;
    int32_t mb;
    int64_t elem_off;   // piece offset inside the channel range (elements)
    int64_t nelem;      // piece length (elements)
    int64_t seq_in;     // first slot sequence number on link_in (per execution)
    int64_t seq_out;    // first slot sequence number on link_out
    int32_t nslots;     // FIFO slots this piece occupies (>= 1 when a link is used)
    int32_t dep_begin;  // waits: deps[dep_begin .. dep_begin + dep_count)
    int32_t dep_count;
    int32_t signal;     // counter to post after the step, or -1
    int32_t flags;      // bit 0: do not post link flags (debug hook); bits 1 / 2: the source /
                        // local operand is an input buffer no instruction writes (streaming loads)
    int32_t drain;      // latest earlier step of the same threadblock whose tiles must be
                        // finished before this step starts (global step index), or -1
};
static_assert(sizeof(DStep) == 64, "DStep layout");

// One segment of a threadblock program: its channel instructions in order,
// run in windows of `window` micro-batches (each instruction takes every
// micro-batch of a window in turn).
struct SegInfo {
    std::vector<int> cis;
    int window = 1;
};

struct PlanImage {
    std::vector<DInstr> instrs;
    std::vector<DStep> steps;
    std::vector<DRec> recs;          // built from instrs + steps at the end of planning
    std::vector<int32_t> tb_begin;   // ntb + 1
    std::vector<DLink> links;
    std::vector<int32_t> prog_links;  // ntb * kSeqLinks: the first links each program uses (-1: none)
    std::vector<DDep> deps;
    std::vector<int32_t> tb_rank;    // rank each threadblock serves (reporting)
    std::vector<std::vector<SegInfo>> tb_segs;   // segments of every threadblock program
    int32_t ntb = 0;
    int32_t ncounters = 0;
    int32_t nthreads = 512;
    int32_t S = 4;
    int64_t slot_bytes = 0;
    int64_t tile_bytes = 0;          // tile of the data path
    int32_t ns = 0;                  // shared-memory stages of the bulk path (set at plan creation)
    int32_t bulk = 0;                // bulk path requested
    int32_t engine = 0;              // CCL_ENGINE_*
    int32_t link_mode = 0;
    int32_t ndirect = 0;             // transfers turned into direct copies
    int32_t channel_scaling = 0;
    int64_t fifo_bytes = 0;
    int32_t m = 1;
    int32_t channels = 1;
    int32_t mb_order = CCL_MB_ALGO;
    int32_t mb_window = 1;           // micro-batches interleaved per instruction inside a segment
    int32_t protocol = 0;            // CCL_PROTO_*: LL slots take 2 x slot_bytes
    int32_t nsubpipelines = 0;
    int32_t ntb_connection = 0;
    int32_t dtype = CCL_F32;
    int32_t esize = 4;
    int64_t chunk_elems = 0;
    int64_t schedule_bytes = 0;
    int64_t min_bytes = 0;
    int64_t data_bytes_per_rank = 0;
    double busbw_factor = 0;
    bool scratch_used[CCL_MAX_RANKS] = {};
    int64_t scratch_elems = 0;       // per rank
    int64_t in_elems = 0, out_elems = 0;
    int32_t timeout_ms = 2000;
    int32_t instrument = 0;
    int32_t fuse = CCL_FUSE_FULL;    // fusion mode of the instructions planned
    int32_t kbuild = 0;              // thread limit of the kernel build launched (512 or 1024; 0: not chosen)
    int32_t cluster = 1;             // CTAs per threadblock program (sequential engine)
};

struct Timeline {
    std::vector<int> sp_lo, sp_hi;   // per instruction: first and last sub-pipeline of its tasks
    std::vector<int> sp_key;         // per instruction: sub-pipeline that orders it in its threadblock
    bool split = false;              // dependencies wait only for the effect task of a fused instruction
    std::vector<int> xfer_sp;        // per transfer
    int nsp = 0;
};

ccl_status_t build_timeline(const ccl_schedule& s, int scheduler, Timeline* tl);

ccl_status_t build_plan(const ccl_schedule& s, int64_t chunk_elems, int32_t dtype,
                        const ccl_plan_opts_t& opts, PlanImage* img);

// Abstract execution of the threadblock programs with bounded FIFOs.
// Returns true when every threadblock finishes; otherwise fills `why`.
bool simulate_plan(const PlanImage& img, std::string* why);

}  // namespace ccl
