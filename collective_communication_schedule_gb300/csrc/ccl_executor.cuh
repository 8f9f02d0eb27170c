// Kernel parameters of the persistent executor: one CTA per threadblock
// program, every rank's buffers and every link FIFO in this GPU's memory.
//
// Each CTA walks its list of (instruction, micro-batch) steps with four
// roles (issuer, releaser, bulk-copy thread, data warps; see
// ccl_runtime.cu).  Per FIFO slot the issuer waits (bounded) until the
// incoming slot is full and the outgoing slot is free, the data path moves
// the slot's data with 16-byte accesses, and the releaser posts the
// consumed / full flags after a gpu-scope release fence.  The flag protocol
// stands in for the inter-GPU links of the pages' runtimes (MSCCLang
// report, §III.1 runtime; ReSCCL report, §II.2 kernel generation).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "ccl_plan.h"

namespace ccl {

struct KParams {
    const DRec* recs;
    const int32_t* tb_begin;
    const DLink* links;
    const DDep* deps;
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
    char* bufs[3][CCL_MAX_RANKS];
};

enum WaitReason : int { WAIT_DEP = 1, WAIT_FULL = 2, WAIT_FREE = 3, WAIT_DONE = 4 };

}  // namespace ccl
