/*
 * ccl.h -- C ABI of the GB300 chunk-schedule collective executor.
 *
 * One GPU holds R *virtual ranks*.  Each rank owns an input, an output and a
 * scratch buffer in HBM; a "link" between two ranks is a FIFO of slots in HBM
 * with per-slot flags, so a transfer is a device-memory copy and no byte
 * leaves the GPU.  A collective is a chunk program (a list of copy / reduce
 * operations on chunk ranges of those buffers) that the host compiles into
 * per-threadblock instruction lists run by one persistent CUDA kernel.
 *
 * Sources of the model (cited by page title and section):
 *   - MSCCLang report (ASPLOS '23), §III.1 "system design": chunk-oriented
 *     programs over input/output/scratch buffers with copy and reduce; the
 *     compiler traces dependencies into a DAG, lowers cross-rank operations
 *     to send/recv/reduce instructions, fuses adjacent ones into
 *     recv-reduce-copy-send style instructions, and spreads them over
 *     channels and threadblocks by a parallelization factor; a runtime
 *     executes the instruction lists with pipelining.
 *   - ReSCCL report (SIGCOMM '25), §II.1-II.2: task-level execution across
 *     micro-batches, hierarchical-priority dynamic scheduling (HPDS) into
 *     sub-pipelines, state-based threadblock allocation.
 *   - AutoCCL report (NSDI '25), "research method" 1-2: resource parameters
 *     nChannel / nThread / chunk size tuned by subspace coordinate descent.
 *
 * Conventions for every function:
 *   - Return CCL_OK or an error code; on error, ccl_last_error_detail()
 *     returns a human-readable reason (thread-local, valid until the next
 *     call on the same thread).  Output handles are left untouched on error.
 *   - Device pointers are CUDA device addresses on the current device.  A
 *     "stream" argument is a cudaStream_t passed as void* (NULL = legacy
 *     default stream).
 *   - Handles (ccl_schedule_t, ccl_plan_t) are owned by the library and freed
 *     by their *_destroy function; nothing returned by the library must be
 *     freed by the caller.
 *   - Nothing here falls back to the CPU: an entry point that needs the GPU
 *     returns CCL_ERR_CUDA when no device or no sm_103 image is usable.
 */
#ifndef CCL_SCHEDULE_H
#define CCL_SCHEDULE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CCL_MAX_RANKS 64

typedef enum {
    CCL_OK = 0,
    CCL_ERR_INVALID_ARG = 1, /* bad argument, out-of-range op, misaligned or overlapping buffers */
    CCL_ERR_CYCLE = 2,       /* dependency cycle among compiled instructions */
    CCL_ERR_DEADLOCK = 3,    /* threadblock programs cannot all finish with the given FIFO capacity */
    CCL_ERR_RACE = 4,        /* two unordered accesses to one buffer range, one of them a write */
    CCL_ERR_UNSUPPORTED = 5, /* valid request the executor cannot run (e.g. threadblocks not co-resident) */
    CCL_ERR_OOM = 6,         /* device allocation failed */
    CCL_ERR_CUDA = 7,        /* a CUDA runtime call failed (no device, launch failure, ...) */
    CCL_ERR_TIMEOUT = 8,     /* a device flag wait ran out of time (reported by ccl_plan_status) */
    CCL_ERR_INTERNAL = 9
} ccl_status_t;

typedef enum { CCL_F32 = 0, CCL_BF16 = 1, CCL_F16 = 2, CCL_I32 = 3 } ccl_dtype_t;
typedef enum { CCL_SUM = 0 } ccl_redop_t;
typedef enum { CCL_BUF_IN = 0, CCL_BUF_OUT = 1, CCL_BUF_SCRATCH = 2 } ccl_buf_t;
typedef enum { CCL_OP_COPY = 0, CCL_OP_REDUCE = 1 } ccl_opcode_t;

/*
 * One chunk operation (MSCCLang report, §III.1): copy  dst := src, or
 * reduce  dst := dst (+) src.  Offsets and counts are in chunks of the
 * buffer kind named by *_buf (ccl_buf_t).  Layout: 8 consecutive int32.
 * Source and destination of one operation must not overlap.
 */
typedef struct {
    int32_t op;       /* ccl_opcode_t */
    int32_t src_rank, src_buf, src_off;
    int32_t dst_rank, dst_buf, dst_off;
    int32_t count;    /* chunks, > 0 */
} ccl_op_t;

typedef struct ccl_schedule* ccl_schedule_t;
typedef struct ccl_plan* ccl_plan_t;

/* Built-in collective programs (ccl_schedule_builtin kinds). */
typedef enum {
    CCL_RING_ALLREDUCE = 0,     /* out[r] = sum_k in[k]; R chunks per buffer */
    CCL_RING_ALLGATHER = 1,     /* out[r] = concat_s in[s]; in 1 chunk, out R chunks */
    CCL_RING_REDUCESCATTER = 2, /* out[r] = chunk r of sum_k in[k]; in R chunks, out 1 chunk */
    CCL_HIER_ALLREDUCE = 3,     /* R = G*ng; intra RS, inter ring AR per slice, intra AG */
    CCL_ALLTOALL_2PHASE = 4,    /* out[d] block s = in[s] block d; R = G*ng */
    CCL_ALLTONEXT = 5,          /* out[r+1] = in[r]; cross-group pairs relayed in G parts */
    CCL_ALLTOALLV = 6           /* uneven AllToAll: built by ccl_schedule_alltoallv only */
} ccl_builtin_t;

#define CCL_FLAG_WRAP 1u    /* AllToNext: also send rank R-1 -> rank 0 */
#define CCL_FLAG_NOFUSE 2u  /* compile without instruction fusion */
/* Fuse as usual but leave a received value that is only copied on (no
 * reduction) as a receive into its buffer plus a send from it, instead of
 * chaining the two into one receive-copy-send; reductions keep their fused
 * forms.  With direct transport each such hop is then one plain copy into
 * the next rank's buffer (the all-gather half of a ring or hierarchical
 * AllReduce). */
#define CCL_FLAG_NOCHAIN_COPIES 4u

/* Fusion modes of ccl_schedule_compile's `fuse` argument. */
#define CCL_FUSE_NONE 0
#define CCL_FUSE_FULL 1
#define CCL_FUSE_NOCHAIN 2  /* as CCL_FLAG_NOCHAIN_COPIES */

/* Fused instruction kinds produced by the compiler (MSCCLang report,
 * §III.1 "instruction generation" and "instruction fusion"). */
typedef enum {
    CCL_I_COPY = 0,      /* dst <- src (one rank) */
    CCL_I_REDUCE = 1,    /* dst <- local (+) src (one rank) */
    CCL_I_SEND = 2,      /* slot_out <- src */
    CCL_I_RECV = 3,      /* dst <- slot_in */
    CCL_I_RRC = 4,       /* dst <- local (+) slot_in           (recv-reduce-copy) */
    CCL_I_RCS = 5,       /* dst <- slot_in; slot_out <- slot_in (recv-copy-send) */
    CCL_I_FWD = 6,       /* slot_out <- slot_in                 (recv-send, relay) */
    CCL_I_RRS = 7,       /* slot_out <- local (+) slot_in       (recv-reduce-send) */
    CCL_I_RRCS = 8,      /* t <- local (+) slot_in; dst <- t; slot_out <- t */
    CCL_I_COPY_SEND = 9, /* dst <- src; slot_out <- src */
    CCL_I_NKINDS = 10,   /* kinds the compiler emits */
    /* plans only (ccl_plan_steps), made by direct transport from a sender
       and the plain receive it feeds (or the copy that forwards it): */
    CCL_I_COPY2 = 10,    /* two-destination copy: dst <- src; loc <- src (a copy-send and its receive, or a
                            chain of two direct copies; loc: the second destination) */
    CCL_I_RRC2 = 11,     /* recv-reduce-copy-send + receive: t <- local (+) slot_in; dst <- t; src <- t
                            (src: the receiver's destination) */
    /* plans only, made by direct transport from two consecutive steps of a
       reduction chain (a send or recv-reduce-send and the receive-reduce
       that its slot feeds), run by the first one's threadblock, which reads
       the second one's local operand itself; the sums keep the chain's
       order, each rounded to the element type: */
    CCL_I_RRS3 = 12,     /* slot_out <- (slot_in (+) local) (+) src  (src: the second step's local) */
    CCL_I_RRC3 = 13,     /* dst <- (slot_in (+) local) (+) src */
    CCL_I_RRCS3 = 14,    /* t <- (slot_in (+) local) (+) src; dst <- t; slot_out <- t */
    CCL_I_RSEND = 15,    /* slot_out <- src (+) local  (a send and the recv-reduce-send it feeds) */
    CCL_I_RCSEND = 16,   /* t <- src (+) local; dst <- t; slot_out <- t  (a send and a recv-reduce-copy-send);
                            a send and the recv-reduce-copy it feeds become a CCL_I_REDUCE */
    /* and with the plain receive that the last two feed folded in (a
       second destination x, the receiver's, instead of the slot): */
    CCL_I_RRC3D = 17,    /* t <- (slot_in (+) local) (+) src; dst <- t; x <- t */
    CCL_I_REDUCE2 = 18,  /* t <- src (+) local; dst <- t; x <- t */
    CCL_I_COPY3 = 19     /* dst <- src; loc <- src; x <- src  (a chain of three direct copies) */
} ccl_instr_kind_t;

typedef struct {
    int32_t nranks;
    int32_t nchunks[3];          /* chunks per rank of in / out / scratch */
    int32_t nops;                /* operations in the source program */
    int32_t ninstr;              /* fused instructions (all ranks) */
    int32_t ntransfers;          /* cross-rank transfers */
    int32_t kind_count[CCL_I_NKINDS];
    int64_t bytes_per_chunk_elem_x_esize; /* schedule bytes = this * chunk_elems * esize */
    int32_t builtin;             /* ccl_builtin_t, or -1 for a compiled program */
    int32_t group_size;
} ccl_schedule_info_t;

/* Per fused instruction, for inspection and tests.  Ranges are in chunks;
 * an absent operand has rank -1. */
typedef struct {
    int32_t kind;                /* ccl_instr_kind_t */
    int32_t rank;
    int32_t src_rank, src_buf, src_off;
    int32_t loc_rank, loc_buf, loc_off;
    int32_t dst_rank, dst_buf, dst_off;
    int32_t count;
    int32_t peer_in;             /* sending rank of the received transfer, or -1 */
    int32_t peer_out;            /* receiving rank of the sent transfer, or -1 */
    int32_t xfer_in, xfer_out;   /* transfer ids, or -1 */
    int32_t position;            /* program position */
} ccl_instr_info_t;

/*
 * Compile a chunk program.  ops[0..nops) in program order; dependencies
 * are traced from program order (read-after-write, write-after-read and
 * write-after-write on overlapping ranges of the same rank's buffer), so the
 * traced DAG is acyclic by construction.  fuse = CCL_FUSE_FULL (or any
 * value other than the two below) applies copy propagation, dead-store
 * elimination and recv/send fusion; CCL_FUSE_NOCHAIN does the same except
 * chaining a copy-only receive into its send; CCL_FUSE_NONE (0) keeps one
 * instruction per half operation.
 * Errors: CCL_ERR_INVALID_ARG (rank/buffer/range out of bounds, count <= 0,
 * overlapping source and destination, nranks outside 1..CCL_MAX_RANKS).
 */
ccl_status_t ccl_schedule_compile(const ccl_op_t* ops, int32_t nops, int32_t nranks,
                                  const int32_t nchunks[3], int32_t fuse, ccl_schedule_t* out);

/*
 * Generate and compile a built-in program.  group_size (G) is used by the
 * hierarchical, AllToAll and AllToNext kinds (nranks must be a multiple of
 * G); the ring kinds ignore it.  flags: CCL_FLAG_WRAP, CCL_FLAG_NOFUSE,
 * CCL_FLAG_NOCHAIN_COPIES (NOFUSE wins when both are set).
 */
ccl_status_t ccl_schedule_builtin(int32_t kind, int32_t nranks, int32_t group_size,
                                  uint32_t flags, ccl_schedule_t* out);

/*
 * Uneven AllToAll (MoE-style token exchange; a variant with per-pair sizes
 * of the AllToAll of the MSCCLang report §IV.3): counts[s * nranks + d] >= 0
 * chunks go from rank s to rank d.  Rank s's input holds its blocks for
 * d = 0, 1, ... in that order (sizes counts[s][d]); rank d's output holds
 * the blocks from s = 0, 1, ... in that order.  Every rank's buffers are as
 * long as the longest rank's (in: max_s sum_d counts[s][d] chunks, out:
 * max_d sum_s counts[s][d]); the tail of a shorter output is not written.
 * One copy per non-empty pair, issued in shift order (d = s + k) so that
 * each round of the program touches distinct links.  flags: CCL_FLAG_NOFUSE,
 * CCL_FLAG_NOCHAIN_COPIES.
 * Errors: CCL_ERR_INVALID_ARG (nranks out of range, a negative count, no
 * chunk to move, a per-rank total above 2^30 chunks).
 */
ccl_status_t ccl_schedule_alltoallv(int32_t nranks, const int32_t* counts, uint32_t flags,
                                    ccl_schedule_t* out);

ccl_status_t ccl_schedule_info(ccl_schedule_t s, ccl_schedule_info_t* info);

/* Copy the source program (ops) or the fused instructions into caller
 * arrays of capacity cap; *n receives the full count (CCL_ERR_INVALID_ARG if
 * cap is too small, after setting *n). */
ccl_status_t ccl_schedule_get_ops(ccl_schedule_t s, ccl_op_t* ops, int32_t cap, int32_t* n);
ccl_status_t ccl_schedule_get_instrs(ccl_schedule_t s, ccl_instr_info_t* out, int32_t cap,
                                     int32_t* n);

void ccl_schedule_destroy(ccl_schedule_t s);

/* Scheduling policies for ccl_plan_opts_t. */
typedef enum { CCL_SCHED_RR = 0, CCL_SCHED_HPDS = 1 } ccl_scheduler_t;
typedef enum { CCL_TB_CONNECTION = 0, CCL_TB_PACKED = 1, CCL_TB_BALANCED = 2 } ccl_tb_alloc_t;
typedef enum { CCL_MB_AUTO = 0, CCL_MB_ALGO = 1, CCL_MB_TASK = 2, CCL_MB_SEGMENT = 3 } ccl_mb_order_t;
typedef enum { CCL_LINK_FIFO = 0, CCL_LINK_DIRECT = 1 } ccl_link_mode_t;
typedef enum { CCL_PROTO_SIMPLE = 0, CCL_PROTO_LL = 1 } ccl_protocol_t;

typedef enum {
    CCL_ENGINE_PIPELINED = 0,    /* warp-specialised CTAs (issuer, data warps, releaser) */
    CCL_ENGINE_SEQUENTIAL = 1    /* one step at a time, every thread moves data */
} ccl_engine_t;

/*
 * Execution parameters of a plan (zero fields take the defaults written by
 * ccl_plan_opts_default).
 *   channels    : parallelization factor; every chunk range is split into
 *                 `channels` contiguous 16-byte-granular pieces, each with its
 *                 own links and threadblocks (MSCCLang report, §III.1, §IV.1).
 *   nthreads    : threads per threadblock (128..1024, multiple of 32: an
 *                 issuing, a releasing and a bulk-copy warp, the rest move
 *                 or add data);
 *                 0 = 512, halved (down to 128) until every threadblock can
 *                 be co-resident.
 *   slot_bytes  : FIFO slot size (multiple of 16).
 *   fifo_slots  : slots per link FIFO (>= 2).
 *   microbatches: pieces every channel range is cut into; 0 = the smallest
 *                 count that keeps a piece within half of a FIFO.
 *   scheduler   : CCL_SCHED_RR (program-order list scheduling) or
 *                 CCL_SCHED_HPDS (ReSCCL report, §II.2).
 *   tb_alloc    : CCL_TB_CONNECTION (one threadblock per (in-link, out-link)
 *                 connection), CCL_TB_PACKED (connections never active in
 *                 the same sub-pipeline share a threadblock), or
 *                 CCL_TB_BALANCED (packed, then the threadblocks that run
 *                 only link-free instructions -- local copies and direct
 *                 copies, which need no FIFO and no particular rank's
 *                 threadblock -- are merged into at most
 *                 max(1, tb_budget / channels) threadblocks of any rank by
 *                 largest-first bin packing on their bytes; for AllToAll-like
 *                 programs with many small or uneven pairs).
 *   mb_order    : order of micro-batches inside a threadblock program.  A
 *                 program is cut into segments run one after the other; a
 *                 segment runs micro-batch-major (each micro-batch through all
 *                 of its instructions).  ALGO cuts only where a dependency on
 *                 a partly overlapping range needs all micro-batches of its
 *                 producer; SEGMENT also cuts at idle gaps of the
 *                 threadblock's sub-pipeline timeline; TASK cuts before every
 *                 instruction (each runs all its micro-batches first:
 *                 task-level execution); AUTO tries ALGO, SEGMENT, TASK in
 *                 that order and keeps the first that can finish.
 *   mb_window   : micro-batches a segment interleaves.  The segment runs its
 *                 micro-batches in windows of this many: each instruction
 *                 of the segment in turn takes every micro-batch of the
 *                 window, so a step has up to mb_window - 1 independent
 *                 pieces ahead of it in its own threadblock while the piece
 *                 it depends on is still in flight upstream.  1 = one
 *                 micro-batch at a time through the whole segment; 0 =
 *                 auto: min(m, fifo_slots / (2 x slots per piece)) first (a
 *                 window and the next one fit in the FIFO together), then 1,
 *                 keeping the first that can finish.
 *   protocol    : FIFO signalling (AutoCCL report: implementation parameter
 *                 "protocol"; MSCCLang report §III.1 runtime protocols).
 *                 CCL_PROTO_SIMPLE: a slot is published by a flag after its
 *                 data (release fence on the sender, flag poll and acquire
 *                 fence on the receiver).  CCL_PROTO_LL: every 4 data bytes
 *                 travel in one 64-bit line with the slot's flag in the high
 *                 half, written and polled with 64-bit accesses (single-copy
 *                 atomic), so the receiver's data path reads the data as soon
 *                 as it lands, with no fence or flag round trip in between;
 *                 a slot occupies 2 x slot_bytes.  LL needs chunk sizes that
 *                 are multiples of 16 bytes, 16-byte aligned buffers and at
 *                 most 512 threads (bulk copies are off); it suits the
 *                 latency-bound sizes.
 *   timeout_ms  : limit of every device flag wait.
 *   instrument  : 1 = record per-step global-timer stamps (ccl_plan_timeline).
 *   tile_bytes  : the executor moves a slot in tiles of this size (multiple of
 *                 16, <= 64 KiB).
 *   bulk        : 1 = move 16-byte-aligned copy tiles through shared memory
 *                 with bulk (TMA) copies; 0 = registers for every tile.
 *   channel_scaling: 1 = an instruction gets a parallelization factor
 *                 proportional to its size (at most `channels`, at least 1),
 *                 so small transfers do not occupy as many threadblocks as
 *                 large ones; 0 = every instruction gets `channels`.
 *   engine      : CCL_ENGINE_PIPELINED (default): warp-specialised CTAs --
 *                 one issuing thread polls the flags of coming steps and
 *                 hands slots to the data warps through shared-memory
 *                 descriptors, one releasing thread posts flags -- so the
 *                 waits of a step overlap the data of earlier ones.
 *                 CCL_ENGINE_SEQUENTIAL: a CTA runs its steps one after
 *                 another; thread 0 waits, every thread moves the slot, a CTA
 *                 barrier, thread 0 fences and posts.  Fewer hand-offs per
 *                 step (for the latency-bound sizes); no bulk copies.  With
 *                 LL every thread polls the lines of its part of an
 *                 incoming slot itself.
 *   link_mode   : transport of a transfer (AutoCCL report: implementation
 *                 parameter "transport").  CCL_LINK_FIFO stages every
 *                 transfer in the link FIFO; CCL_LINK_DIRECT lets a plain
 *                 send from a buffer write straight into the receiver's
 *                 destination buffer (one copy, no FIFO) and keeps FIFOs for
 *                 transfers that are forwarded or reduced.
 *   cluster     : sequential engine only: run every threadblock program on a
 *                 thread-block cluster of this many CTAs (2, 4 or 8).  Every
 *                 CTA waits for the step's flags and counters itself and
 *                 moves its 16-byte-granular share of each slot; after one
 *                 cluster barrier the cluster's first CTA posts.  Same steps,
 *                 channels and FIFOs (one program per channel); the data of a
 *                 step moves on `cluster` SMs instead of one, for the
 *                 latency-bound sizes where a single CTA's data time sets the
 *                 length of every hop.
 *   fold        : with direct transport, a bit mask (default 3).
 *                 Bit 0 (1): a plain receive fed by a copy-send or a
 *                 recv-reduce-copy-send is folded into its sender, whose
 *                 pass then writes the receiver's buffer too (CCL_I_COPY2 /
 *                 CCL_I_RRC2 steps; one step and 2 bytes per element byte
 *                 fewer per such pair); cleared, such senders keep their
 *                 FIFO.  Bit 1 (2): copy chains -- a direct copy that sends
 *                 on, unchanged, exactly the range another direct copy
 *                 delivered is run by that copy's pass (a CCL_I_COPY2 with
 *                 two remote destinations: one read written twice, 3 bytes
 *                 per element byte instead of 2 + 2, one step fewer); a
 *                 chain of k copies from its head becomes ceil(k/2) steps,
 *                 and a pair whose merged dependencies would cycle is kept
 *                 apart.  Bit 2 (4): reduction chains -- a send or
 *                 recv-reduce-send and the receive-reduce its slot feeds
 *                 run as one step on the first one's threadblock, which
 *                 reads the second rank's local operand itself and adds it
 *                 after its own sum (the chain's order and rounding; the
 *                 CCL_I_RSEND, RCSEND, RRS3, RRC3, RRCS3 steps, or a
 *                 CCL_I_REDUCE across ranks): the slot between them (2
 *                 bytes per element byte) and a hop go, and the step sends
 *                 on where the second one sent; with bit 0 the plain
 *                 receive such a step feeds is folded into it as a second
 *                 destination (CCL_I_RRC3D, CCL_I_REDUCE2); not with the LL
 *                 protocol.  Bit 3 (8): copy chains three hops per step
 *                 (CCL_I_COPY3, its third destination in the fourth range:
 *                 one read written three times, 4 bytes per element byte
 *                 instead of 2 + 2 + 2).  Bit 2 is not in the
 *                 default: where a chain's other hops stay one rank apart
 *                 (a fully fused ring AllReduce's all-gather) a rank then
 *                 needs links one and two ranks away and more
 *                 threadblocks; with the all-gather hops direct (copy
 *                 receives unchained) it does not.  A folded plan
 *                 that would cycle or deadlock is planned again without
 *                 folds.  Values outside 0..15: CCL_ERR_INVALID_ARG.
 *   codegen     : 0 (default): the library's kernels interpret the plan's
 *                 step records.  1: ccl_plan_create generates CUDA source
 *                 for this one plan (ReSCCL report, §II.2: a kernel per
 *                 schedule instead of a run-time interpreter), compiles it
 *                 for sm_103a with NVRTC and runs it instead: every
 *                 threadblock program becomes code with its instructions'
 *                 buffers, offsets, links and counters written in, and no
 *                 step, link or dependency table is read on the device.
 *                 Same steps, waits, status word and results as the
 *                 interpreted plan.  Identical generated sources are compiled
 *                 once per process.  Flag protocol only; a plan whose steps
 *                 the generator cannot express as loops is refused
 *                 (CCL_ERR_UNSUPPORTED), so is ccl_plan_debug_drop_signal on
 *                 a generated plan.
 */
typedef struct {
    int32_t channels;
    int32_t nthreads;
    int64_t slot_bytes;
    int32_t fifo_slots;
    int32_t microbatches;
    int32_t scheduler;
    int32_t tb_alloc;
    int32_t mb_order;
    int32_t timeout_ms;
    int32_t instrument;
    int64_t tile_bytes;
    int32_t bulk;
    int32_t link_mode;
    int32_t channel_scaling;
    int32_t mb_window;
    int32_t protocol;
    int32_t tb_budget;   /* CCL_TB_BALANCED: threadblocks to aim for (0: 256) */
    int32_t engine;      /* CCL_ENGINE_* */
    int32_t codegen;     /* 1: run a kernel generated and compiled for this plan (see below) */
    int32_t cluster;     /* sequential engine: CTAs per threadblock program (0 or 1: one; 2, 4, 8) */
    int32_t fold;        /* direct transport: bit 0 folds plain receives into their senders, bit 1
                            copy chains, bit 2 reduction chains, bit 3 three-hop copy chains (default 3) */
} ccl_plan_opts_t;

void ccl_plan_opts_default(ccl_plan_opts_t* o);

/*
 * Build an executable plan for `chunk_elems` elements per chunk.  Rank r's
 * input buffer then holds nchunks[0] * chunk_elems elements, its output
 * nchunks[1] * chunk_elems.  Allocates (library-owned, on the current
 * device): link FIFOs and flags, scratch for ranks whose scratch is touched,
 * and the instruction tables.  Validates the threadblock programs by
 * simulating them (CCL_ERR_DEADLOCK) and checks that all threadblocks can be
 * co-resident (CCL_ERR_UNSUPPORTED).  dtype: ccl_dtype_t; op: CCL_SUM.
 * A fused schedule whose instructions cannot be planned with these options
 * (a fused send keeps more transfers in flight on a link than the FIFO
 * holds, or no task order exists) is planned from the same program compiled
 * with less fusion (copy receives unchained, then none): same results, more
 * bytes; ccl_plan_stats reports the mode used.
 */
ccl_status_t ccl_plan_create(ccl_schedule_t s, int64_t chunk_elems, int32_t dtype, int32_t op,
                             const ccl_plan_opts_t* opts, ccl_plan_t* out);

/*
 * Run the plan on `stream` (asynchronous).  in_bufs[r] / out_bufs[r] are
 * device pointers to rank r's input / output (16-byte alignment gives the
 * vector path; any element-aligned pointer is accepted).  An input may equal
 * its rank's output only if the program never reads that rank's input after
 * writing its output; other overlaps between buffers are the caller's
 * responsibility.  Launch errors return CCL_ERR_CUDA; a device timeout is
 * reported later by ccl_plan_status.  A plan must not run concurrently with
 * itself (one stream at a time).
 */
ccl_status_t ccl_execute(ccl_plan_t p, void* const* in_bufs, void* const* out_bufs, void* stream);

/*
 * End-to-end form: copy host_in[r] (host memory; pinned gives asynchronous
 * copies) to dev_in[r], run the plan, copy dev_out[r] back to host_out[r],
 * all on `stream`.  The caller synchronizes the stream before reading
 * host_out.
 */
ccl_status_t ccl_execute_host(ccl_plan_t p, const void* const* host_in, void* const* host_out,
                              void* const* dev_in, void* const* dev_out, void* stream);

/*
 * End-to-end form over three streams, for pipelining several plans: the
 * input copies go on copy_in_stream, the kernel on compute_stream after them,
 * the output copies on copy_out_stream after the kernel (events owned by the
 * plan, created on its first such call).  Host-to-device and device-to-host
 * copies then overlap across plans that share the three streams.  A later
 * call with the same plan orders its input copies after this call's kernel
 * and its kernel after this call's output copies, so the plan's device
 * buffers may be reused from call to call; mixing this call with
 * ccl_execute on the same buffers needs the caller's own ordering.  The
 * caller synchronizes copy_out_stream before reading host_out.
 */
ccl_status_t ccl_execute_host_async(ccl_plan_t p, const void* const* host_in, void* const* host_out,
                                    void* const* dev_in, void* const* dev_out, void* copy_in_stream,
                                    void* compute_stream, void* copy_out_stream);

/*
 * Status of the last execution, to call after synchronizing its stream:
 * CCL_OK, or CCL_ERR_TIMEOUT when a flag wait ran out (the detail names the
 * threadblock and step).  After a timeout the plan's flags are reset so the
 * plan can run again.
 */
ccl_status_t ccl_plan_status(ccl_plan_t p);

typedef struct {
    int64_t schedule_bytes;      /* bytes read + written by all fused instructions per execution */
    int64_t min_bytes;           /* inputs read once + outputs written once */
    int64_t data_bytes_per_rank; /* message size used for algBW (per builtin kind) */
    double busbw_factor;         /* nccl-tests convention: algBW -> busBW */
    int32_t nthreadblocks;       /* threadblocks in the launch */
    int32_t nthreadblocks_connection; /* count under one-threadblock-per-connection */
    int32_t nsteps;              /* (instruction, micro-batch) steps over all threadblocks */
    int32_t ninstr;              /* channel instructions */
    int32_t nlinks;              /* link FIFOs */
    int32_t nsubpipelines;       /* sub-pipelines of the scheduler's timeline */
    int32_t microbatches;
    int32_t mb_order;            /* order actually used */
    int32_t channels, nthreads, fifo_slots;
    int64_t slot_bytes;
    int64_t fifo_bytes;          /* device bytes of all link FIFOs */
    int64_t device_bytes;        /* all device memory owned by the plan */
    double compile_ms;           /* host time of ccl_plan_create */
    int64_t tile_bytes;          /* tile of the data path */
    int32_t stages;              /* shared-memory stages of the bulk path (0: registers only) */
    int32_t mb_window;           /* micro-batch window actually used */
    int32_t protocol;            /* CCL_PROTO_* */
    int32_t engine;              /* CCL_ENGINE_* */
    int32_t fuse;                /* CCL_FUSE_* mode of the instructions planned (less than the
                                    schedule's when its fused form could not be planned) */
    int32_t kernel_build;        /* thread limit the launched kernel was built for: 512 (eight
                                    16-byte vectors in flight per thread) or 1024 (four); 0 from
                                    ccl_plan_check, which does not choose */
    int32_t cluster;             /* CTAs per threadblock program (1 unless the sequential engine runs
                                    on clusters) */
    int32_t codegen;             /* 1: the plan runs its generated kernel */
    double codegen_ms;           /* host time to generate and compile it (0 when cached) */
} ccl_plan_stats_t;

ccl_status_t ccl_plan_stats(ccl_plan_t p, ccl_plan_stats_t* st);

/*
 * The CUDA source ccl_plan_create would generate for this schedule, size and
 * options with codegen = 1 (host only, no device needed): copied into buf
 * (capacity cap bytes, NUL-terminated) unless buf is NULL; *len (may be
 * NULL) receives its length without the NUL.  With compile = 1 the source
 * is also compiled for sm_103a with NVRTC and *cubin_bytes (may be NULL)
 * receives the size of the result.  The kernel is built for 512 threads
 * when opts->nthreads <= 512, else for 1024.  Errors: those of
 * ccl_plan_check, CCL_ERR_UNSUPPORTED (the generator cannot express the
 * plan), CCL_ERR_INVALID_ARG (cap too small, after setting *len),
 * CCL_ERR_INTERNAL (the compiler rejected the source; the detail holds its
 * log).
 */
ccl_status_t ccl_plan_codegen_source(ccl_schedule_t s, int64_t chunk_elems, int32_t dtype,
                                     const ccl_plan_opts_t* opts, char* buf, size_t cap, size_t* len,
                                     int32_t compile, int64_t* cubin_bytes);

/*
 * Run the planner and its deadlock simulation on the host only (no device
 * memory, no GPU needed) and report what ccl_plan_create would build.
 * Returns the same validation errors as ccl_plan_create except the
 * co-residency check (CCL_ERR_UNSUPPORTED), which needs the device.
 */
ccl_status_t ccl_plan_check(ccl_schedule_t s, int64_t chunk_elems, int32_t dtype,
                            const ccl_plan_opts_t* opts, ccl_plan_stats_t* st);

/*
 * Sub-pipeline timeline of a schedule (ReSCCL report, §II.2): xfer_sp[x]
 * receives the sub-pipeline of transfer x (array of ccl_schedule_info_t
 * .ntransfers entries, may be NULL) and *nsub the number of sub-pipelines.
 * scheduler: CCL_SCHED_RR or CCL_SCHED_HPDS.
 */
ccl_status_t ccl_schedule_timeline(ccl_schedule_t s, int32_t scheduler, int32_t* xfer_sp, int32_t* nsub);

/*
 * Threadblock utilisation of the last execution of an instrumented plan
 * (ReSCCL report, §III: mean and maximum threadblock idle rate).  For each
 * threadblock b: busy[b] = length of the union, over its steps, of the
 * interval from the end of the step's waits to the post of its last tile
 * (steps of one threadblock overlap); span = first start to last end over
 * all threadblocks; idle[b] = 1 - busy[b] / span.  Arrays of capacity cap
 * (>= nthreadblocks).  Synchronizes the device.
 */
ccl_status_t ccl_plan_timeline(ccl_plan_t p, double* idle, int32_t cap, double* mean_idle,
                               double* max_idle, double* span_us);

/*
 * Raw stamps of the last execution of an instrumented plan, five per step
 * in threadblock-program order: the global-timer time (ns) the issuer took
 * the step up; the ns it spent waiting for dependency counters and FIFO
 * flags; the time it handed out the step's first tile; the time the
 * releasing warp saw the step's last tile finished (before its release
 * fence); the time that tile's flags were posted.  stamps: capacity cap
 * (>= 5 * nsteps) or NULL; tb_begin: capacity tb_cap (>= nthreadblocks
 * + 1) or NULL, the first step of every threadblock; *nsteps (may be NULL)
 * receives the step count.  With stamps non-NULL the plan must have been
 * created with instrument = 1; synchronizes the device.
 */
ccl_status_t ccl_plan_timeline_raw(ccl_plan_t p, uint64_t* stamps, int64_t cap, int32_t* tb_begin,
                                   int32_t tb_cap, int64_t* nsteps);

/* One step of a threadblock program: one channel piece of one fused
 * instruction for one micro-batch. */
typedef struct {
    int32_t tb;          /* threadblock that runs it */
    int32_t kind;        /* CCL_I_* */
    int32_t rank;        /* rank the threadblock serves */
    int32_t channel;
    int32_t mb;          /* micro-batch */
    int32_t link_in;     /* incoming link FIFO of the plan, or -1 */
    int32_t link_out;    /* outgoing link FIFO, or -1 */
    int32_t nslots;      /* FIFO slots the piece occupies (0: no link) */
    int32_t dep_count;   /* counters waited on before it starts */
    int32_t drain;       /* earlier step of the same threadblock it follows, or -1 */
    int64_t nelem;       /* elements of the piece */
} ccl_step_info_t;

/*
 * The steps of a plan in threadblock-program order (the order of the stamps
 * of ccl_plan_timeline_raw).  out: capacity cap, or NULL to ask for *n only.
 * CCL_ERR_INVALID_ARG when cap is too small (after setting *n).
 */
ccl_status_t ccl_plan_steps(ccl_plan_t p, ccl_step_info_t* out, int64_t cap, int64_t* n);

/*
 * Test hook: make threadblock `tb` skip the FIFO flag posts and the
 * dependency-counter post of its step `step` (the data is still written),
 * so a peer's wait runs out.  Used to check that a lost signal ends in
 * CCL_ERR_TIMEOUT with a usable device.
 */
ccl_status_t ccl_plan_debug_drop_signal(ccl_plan_t p, int32_t tb, int32_t step);

void ccl_plan_destroy(ccl_plan_t p);

/* Tuner (AutoCCL report, "research method" 2: subspace coordinate descent
 * over nChannel, nThread, chunk size, raising each while bandwidth
 * improves). */
typedef struct {
    int32_t max_rounds;          /* coordinate sweeps (default 3) */
    int32_t reps;                /* timed executions per probe; the median is used (default 5) */
    double min_gain;             /* relative improvement to keep moving (default 0.01) */
    int32_t max_channels;        /* largest channel count searched (0: the whole grid) */
} ccl_tune_opts_t;

typedef struct {
    int32_t probes;              /* configurations timed */
    double best_us;              /* median time of the chosen configuration */
    double best_gbs;             /* schedule bytes / best_us */
    double default_us;           /* median time of the default configuration */
} ccl_tune_report_t;

/*
 * Tune channels, threads and slot size for one schedule and size by timing
 * executions on the caller's buffers (their contents are overwritten).
 * `start` (nullable) is the first point; `best` receives the result.
 */
ccl_status_t ccl_tune(ccl_schedule_t s, int64_t chunk_elems, int32_t dtype,
                      void* const* in_bufs, void* const* out_bufs, void* stream,
                      const ccl_tune_opts_t* topts, const ccl_plan_opts_t* start,
                      ccl_plan_opts_t* best, ccl_tune_report_t* report);

/*
 * Ring AllReduce that allocates nothing.  The pages have no counterpart of
 * this call; it is here for callers that must not allocate device memory when
 * they run a collective (all device memory already reserved by a framework
 * allocator, no room for the device-wide synchronisation a cudaMalloc may
 * cause mid-step, or a policy of no allocation after start-up).
 *
 * Computes out_bufs[r] = sum_k in_bufs[k] for r < nranks, each rank buffer
 * holding nranks * chunk_elems elements of `dtype`, with the same fused ring
 * program and therefore the same reduction order (bit for bit) as a plan
 * built from ccl_schedule_builtin(CCL_RING_ALLREDUCE).  channels: 0 picks
 * min(8, 64 / nranks).
 *
 * Memory: the link FIFOs (4 slots of 32 KiB per link), flags and a status
 * word live in one file-scope device array of 8 MiB + 4160 bytes.  The
 * device backs it when it loads the library's device code: with CUDA's
 * default lazy module loading that is the first call of this function on
 * each device (at library load only when modules load eagerly); from then
 * on that GPU holds it until the process exits.  nranks * channels may not
 * exceed 64 links (CCL_ERR_INVALID_ARG otherwise).  This call makes no
 * cudaMalloc, cudaFree or other allocating call, on the host or the device.
 *
 * The first call on a device also looks up the array's device address with
 * cudaGetSymbolAddress (once per device, that device current); make that
 * first call before any stream capture, and outside any latency-critical
 * step.  Every call clears the flags on `stream` and launches one
 * cooperative kernel; all calls share the array, so calls whose executions
 * overlap on the GPU (other streams, other host threads) race and corrupt
 * each other: serialise them.  in_bufs[r] may equal out_bufs[r] (in place).
 * A device wait that runs out of time (2 s) leaves the outputs incomplete;
 * this call does not report it (use the plan API when that matters).
 * Returns CCL_OK, CCL_ERR_INVALID_ARG, CCL_ERR_UNSUPPORTED or CCL_ERR_CUDA.
 */
ccl_status_t ccl_allreduce_ring_noalloc(void* const* in_bufs, void* const* out_bufs, int32_t nranks,
                                        int64_t chunk_elems, int32_t dtype, int32_t channels, void* stream);

/*
 * The search of ccl_tune on its own (AutoCCL report, research method 1-2):
 * the implementation parameters threadblock policy (connection / balanced)
 * x protocol (simple / LL) x transport (FIFO / direct) x engine (pipelined
 * / sequential) make sixteen subspaces; in each, coordinate descent over
 * channels, threads and slot size (and CTAs per program on the sequential
 * engine, and each fold bit with direct transport), driven by a
 * caller-supplied probe that returns the bandwidth of a configuration (any
 * unit, <= 0 = cannot run).  start (nullable) is the first point; best gets
 * the winner, *best_bw its bandwidth, *probes the number of distinct
 * configurations probed.  Host only; no device is touched unless the probe
 * does.
 */
ccl_status_t ccl_tune_search(const ccl_plan_opts_t* start, const ccl_tune_opts_t* topts,
                             double (*probe)(void* user, const ccl_plan_opts_t* o), void* user,
                             ccl_plan_opts_t* best, double* best_bw, int32_t* probes);

/* One row of a per-size tuning table. */
typedef struct {
    int64_t chunk_elems;         /* message size of the row (elements per chunk) */
    ccl_plan_opts_t best;        /* configuration chosen for it */
    ccl_tune_report_t report;    /* its timings */
} ccl_tune_row_t;

/*
 * Tune one schedule for several message sizes (AutoCCL report, research
 * method 1-2: parameters chosen per message size): rows[i] (caller array of
 * n) receives ccl_tune's result for chunk_elems[i].  in_bufs / out_bufs must
 * hold the largest size (their contents are overwritten).  Stops at the
 * first size that cannot be tuned and returns its error.
 */
ccl_status_t ccl_tune_table(ccl_schedule_t s, int32_t dtype, const int64_t* chunk_elems, int32_t n,
                            void* const* in_bufs, void* const* out_bufs, void* stream,
                            const ccl_tune_opts_t* topts, const ccl_plan_opts_t* start, ccl_tune_row_t* rows);

/*
 * Tuning tables as JSON files ("ccl-tune-table-1": dtype, a free-text note,
 * one row per size with the chosen plan options by field name and the
 * timings).  Reading with rows = NULL only sets *n (and *dtype); otherwise
 * cap must be >= the row count.  Fields missing from a row take
 * ccl_plan_opts_default's values.  Errors: CCL_ERR_INVALID_ARG (file cannot
 * be opened or written, malformed content, capacity too small).
 */
ccl_status_t ccl_tune_table_write_json(const ccl_tune_row_t* rows, int32_t n, int32_t dtype, const char* note,
                                       const char* path);
ccl_status_t ccl_tune_table_read_json(const char* path, ccl_tune_row_t* rows, int32_t cap, int32_t* n,
                                      int32_t* dtype);

/* The options of the row whose size is nearest to chunk_elems (ratio of
 * sizes closest to 1; the first of equals). */
ccl_status_t ccl_tune_table_lookup(const ccl_tune_row_t* rows, int32_t n, int64_t chunk_elems,
                                   ccl_plan_opts_t* out);

/*
 * A compiled schedule as a JSON file ("ccl-schedule-1": the source program,
 * chunk counts, fusion mode, built-in kind and a digest of the fused
 * instructions), for checkpointing and reuse.  Reading compiles the program
 * again and fails with CCL_ERR_INVALID_ARG when the instructions differ from
 * the written digest (a compiler that fuses differently), or when the file
 * cannot be read or parsed; the new handle is the caller's to destroy.
 */
ccl_status_t ccl_schedule_write_json(ccl_schedule_t s, const char* path);
ccl_status_t ccl_schedule_read_json(const char* path, ccl_schedule_t* out);

const char* ccl_error_string(ccl_status_t s);
const char* ccl_last_error_detail(void);
const char* ccl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CCL_SCHEDULE_H */
