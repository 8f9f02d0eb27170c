// Memory layout shared by the host planner, the executor kernels built with
// the library and the kernels generated for single plans at run time (which
// are compiled without any standard or C ABI header): the per-step records,
// links, dependency waits and kernel parameters, and the codes of the C ABI
// that device code uses.  Plain C++ (no CUDA keywords, no includes).
#pragma once

#ifndef CCL_SCHEDULE_H
// Without include/ccl.h (run-time compilation): the codes device code needs,
// with the values the C ABI gives them (a host test compares the two).
enum { CCL_F32 = 0, CCL_BF16 = 1, CCL_F16 = 2, CCL_I32 = 3 };
enum { CCL_BUF_IN = 0, CCL_BUF_OUT = 1, CCL_BUF_SCRATCH = 2 };
enum {
    CCL_I_COPY = 0, CCL_I_REDUCE = 1, CCL_I_SEND = 2, CCL_I_RECV = 3, CCL_I_RRC = 4,
    CCL_I_RCS = 5, CCL_I_FWD = 6, CCL_I_RRS = 7, CCL_I_RRCS = 8, CCL_I_COPY_SEND = 9, CCL_I_COPY2 = 10,
    CCL_I_RRC2 = 11, CCL_I_RRS3 = 12, CCL_I_RRC3 = 13, CCL_I_RRCS3 = 14, CCL_I_RSEND = 15, CCL_I_RCSEND = 16,
    CCL_I_RRC3D = 17, CCL_I_REDUCE2 = 18, CCL_I_COPY3 = 19
};
enum { CCL_ERR_TIMEOUT = 8 };
#define CCL_MAX_RANKS 64
#endif

namespace ccl {

// DStep / DRec flags
enum : int { STEP_NOPOST = 1, STEP_SRC_STREAM = 2, STEP_LOC_STREAM = 4 };

// what a failed wait was waiting for (status word [3])
enum WaitReason : int { WAIT_DEP = 1, WAIT_FULL = 2, WAIT_FREE = 3, WAIT_DONE = 4 };

// Everything the executor needs for one step, denormalised (one 144-byte
// record per step, prefetched as one group of 16-byte asynchronous copies).
struct DRec {
    int kind, dtype, link_in, link_out;
    int src_buf, src_rank, loc_buf, loc_rank, dst_buf, dst_rank;
    int nslots, dep_begin, dep_count, signal, mb, flags;
    long long src_off, loc_off, dst_off;   // element offsets of this piece
    long long nelem, seq_in, seq_out;
    int drain;
    int seq_in_mod, seq_out_mod;   // seq_in % S, seq_out % S (slot index arithmetic in 32 bits)
    int link_loc;                  // 1 + the incoming (bits 0-7) and outgoing (bits 8-15) link's entry in
                                   // its program's link table (KParams.prog_links); 0: read the link array
    int x_buf, x_rank;             // a second destination (a folded receive of a three-operand or
    long long x_off;               // cross-rank reduce step), buf -1 when none
};
static_assert(sizeof(DRec) == 144, "DRec layout");

struct DLink {
    long long slot_base;  // byte offset of slot 0 in the FIFO pool (slots of slot_stride bytes)
    long long total;      // slot sequences per execution
    int flag_base;        // full flags at [flag_base, +S), consumed at [flag_base+S, +S)
    int src_rank, dst_rank;
    int total_mod;        // total % S
};
static_assert(sizeof(DLink) == 32, "DLink layout");

struct DDep {
    int counter;
    int pad;
    long long value;      // wait until counter >= exec * m + value
};
static_assert(sizeof(DDep) == 16, "DDep layout");

// links a threadblock program keeps in shared memory (the sequential
// engine); a program's further links are read from the link array
constexpr int kSeqLinks = 8;

// Kernel parameters of the persistent executor: one CTA per threadblock
// program, every rank's buffers and every link FIFO in this GPU's memory.
struct KParams {
    const DRec* recs;
    const int* tb_begin;
    const DLink* links;
    const DDep* deps;
    const int* prog_links;         // kSeqLinks link indices per threadblock program (-1: none)
    unsigned long long* flags;
    unsigned long long* counters;
    char* fifo;
    int* status;                   // [0] code, [1] threadblock, [2] step, [3] reason
    unsigned long long* timeline;  // 5 stamps per step, or null
    long long exec;
    long long m;
    long long slot_bytes;          // data bytes of a slot
    long long slot_stride;         // bytes a slot occupies (2 x slot_bytes for LL)
    unsigned long long timeout_ns;
    long long tile_bytes;          // bytes per tile handed to the data path
    int S;
    int ns;                        // shared-memory stages of the bulk path (0: off)
    int ll;                        // FIFO slots hold LL lines (data + flag per 64 bits)
    int stream_in;                 // inputs share no memory with outputs: streaming loads allowed
    int cluster;                   // sequential engine: CTAs (one thread-block cluster) per threadblock program
    char* bufs[3][CCL_MAX_RANKS];
};

}  // namespace ccl
