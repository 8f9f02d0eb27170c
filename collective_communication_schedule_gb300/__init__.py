"""GB300 executor for chunk-oriented collective schedules (Python binding).

Thin ctypes binding over ``libccl.so`` (C ABI in ``include/ccl.h``): argument
marshalling only.  Every step of the collective runs in the library's CUDA
kernel; PyTorch supplies device memory and streams.  Importing this package
fails loudly when the library has not been built -- there is no CPU path.

    import collective_communication_schedule_gb300 as ccl
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, nranks=8)
    p = ccl.Plan(s, chunk_elems=32768, dtype=ccl.F32, channels=4)
    p.execute(inputs, outputs)          # lists of torch CUDA tensors
    p.status()                          # raises on a device timeout
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libccl.so")

F32, BF16, F16, I32 = 0, 1, 2, 3
IN, OUT, SCRATCH = 0, 1, 2
COPY, REDUCE = 0, 1
RING_ALLREDUCE, RING_ALLGATHER, RING_REDUCESCATTER, HIER_ALLREDUCE, ALLTOALL_2PHASE, ALLTONEXT, ALLTOALLV = range(7)
FLAG_WRAP, FLAG_NOFUSE, FLAG_NOCHAIN_COPIES = 1, 2, 4
FUSE_NONE, FUSE_FULL, FUSE_NOCHAIN = 0, 1, 2
SCHED_RR, SCHED_HPDS = 0, 1
TB_CONNECTION, TB_PACKED, TB_BALANCED = 0, 1, 2
MB_AUTO, MB_ALGO, MB_TASK, MB_SEGMENT = 0, 1, 2, 3
LINK_FIFO, LINK_DIRECT = 0, 1
PROTO_SIMPLE, PROTO_LL = 0, 1
ENGINE_PIPELINED, ENGINE_SEQUENTIAL = 0, 1
KIND_NAMES = ["copy", "reduce", "send", "recv", "rrc", "rcs", "fwd", "rrs", "rrcs", "copy_send", "copy2", "rrc2",
              "rrs3", "rrc3", "rrcs3", "rsend", "rcsend", "rrc3d", "reduce2", "copy3"]
DTYPE_NAMES = {F32: "f32", BF16: "bf16", F16: "f16", I32: "i32"}
ESIZE = {F32: 4, BF16: 2, F16: 2, I32: 4}

STATUS = {0: "ok", 1: "invalid argument", 2: "dependency cycle", 3: "deadlock", 4: "data race",
          5: "unsupported", 6: "out of device memory", 7: "CUDA error", 8: "device wait timed out",
          9: "internal error"}


class CclError(RuntimeError):
    def __init__(self, code, detail):
        super().__init__(f"{STATUS.get(code, code)}: {detail}")
        self.code = code
        self.detail = detail


class Op(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("op", "src_rank", "src_buf", "src_off", "dst_rank", "dst_buf", "dst_off", "count")]


class ScheduleInfo(ctypes.Structure):
    _fields_ = [("nranks", ctypes.c_int32), ("nchunks", ctypes.c_int32 * 3), ("nops", ctypes.c_int32),
                ("ninstr", ctypes.c_int32), ("ntransfers", ctypes.c_int32),
                ("kind_count", ctypes.c_int32 * 10), ("bytes_per_chunk_elem_x_esize", ctypes.c_int64),
                ("builtin", ctypes.c_int32), ("group_size", ctypes.c_int32)]


class InstrInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("kind", "rank", "src_rank", "src_buf", "src_off", "loc_rank", "loc_buf", "loc_off",
                 "dst_rank", "dst_buf", "dst_off", "count", "peer_in", "peer_out", "xfer_in", "xfer_out",
                 "position")]


class PlanOpts(ctypes.Structure):
    _fields_ = [("channels", ctypes.c_int32), ("nthreads", ctypes.c_int32), ("slot_bytes", ctypes.c_int64),
                ("fifo_slots", ctypes.c_int32), ("microbatches", ctypes.c_int32), ("scheduler", ctypes.c_int32),
                ("tb_alloc", ctypes.c_int32), ("mb_order", ctypes.c_int32), ("timeout_ms", ctypes.c_int32),
                ("instrument", ctypes.c_int32), ("tile_bytes", ctypes.c_int64), ("bulk", ctypes.c_int32),
                ("link_mode", ctypes.c_int32), ("channel_scaling", ctypes.c_int32), ("mb_window", ctypes.c_int32),
                ("protocol", ctypes.c_int32), ("tb_budget", ctypes.c_int32), ("engine", ctypes.c_int32),
                ("codegen", ctypes.c_int32), ("cluster", ctypes.c_int32), ("fold", ctypes.c_int32)]


class PlanStats(ctypes.Structure):
    _fields_ = [("schedule_bytes", ctypes.c_int64), ("min_bytes", ctypes.c_int64),
                ("data_bytes_per_rank", ctypes.c_int64), ("busbw_factor", ctypes.c_double),
                ("nthreadblocks", ctypes.c_int32), ("nthreadblocks_connection", ctypes.c_int32),
                ("nsteps", ctypes.c_int32), ("ninstr", ctypes.c_int32), ("nlinks", ctypes.c_int32),
                ("nsubpipelines", ctypes.c_int32), ("microbatches", ctypes.c_int32), ("mb_order", ctypes.c_int32),
                ("channels", ctypes.c_int32), ("nthreads", ctypes.c_int32), ("fifo_slots", ctypes.c_int32),
                ("slot_bytes", ctypes.c_int64), ("fifo_bytes", ctypes.c_int64), ("device_bytes", ctypes.c_int64),
                ("compile_ms", ctypes.c_double), ("tile_bytes", ctypes.c_int64), ("stages", ctypes.c_int32),
                ("mb_window", ctypes.c_int32), ("protocol", ctypes.c_int32), ("engine", ctypes.c_int32),
                ("fuse", ctypes.c_int32), ("kernel_build", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("codegen", ctypes.c_int32), ("codegen_ms", ctypes.c_double)]


class StepInfo(ctypes.Structure):
    _fields_ = [("tb", ctypes.c_int32), ("kind", ctypes.c_int32), ("rank", ctypes.c_int32), ("channel", ctypes.c_int32),
                ("mb", ctypes.c_int32), ("link_in", ctypes.c_int32), ("link_out", ctypes.c_int32),
                ("nslots", ctypes.c_int32), ("dep_count", ctypes.c_int32), ("drain", ctypes.c_int32),
                ("nelem", ctypes.c_int64)]


class TuneOpts(ctypes.Structure):
    _fields_ = [("max_rounds", ctypes.c_int32), ("reps", ctypes.c_int32), ("min_gain", ctypes.c_double),
                ("max_channels", ctypes.c_int32)]


class TuneReport(ctypes.Structure):
    _fields_ = [("probes", ctypes.c_int32), ("best_us", ctypes.c_double), ("best_gbs", ctypes.c_double),
                ("default_us", ctypes.c_double)]


class TuneRow(ctypes.Structure):
    _fields_ = [("chunk_elems", ctypes.c_int64), ("best", PlanOpts), ("report", TuneReport)]


PROBE_FN = ctypes.CFUNCTYPE(ctypes.c_double, ctypes.c_void_p, ctypes.POINTER(PlanOpts))


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
    L = ctypes.CDLL(_LIB_PATH)
    P, I32_, I64_, U32_ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
    sig = {
        "ccl_schedule_compile": [ctypes.POINTER(Op), I32_, I32_, ctypes.POINTER(ctypes.c_int32), I32_,
                                 ctypes.POINTER(P)],
        "ccl_schedule_builtin": [I32_, I32_, I32_, U32_, ctypes.POINTER(P)],
        "ccl_schedule_alltoallv": [I32_, ctypes.POINTER(ctypes.c_int32), U32_, ctypes.POINTER(P)],
        "ccl_schedule_info": [P, ctypes.POINTER(ScheduleInfo)],
        "ccl_schedule_get_ops": [P, ctypes.POINTER(Op), I32_, ctypes.POINTER(ctypes.c_int32)],
        "ccl_schedule_get_instrs": [P, ctypes.POINTER(InstrInfo), I32_, ctypes.POINTER(ctypes.c_int32)],
        "ccl_plan_create": [P, I64_, I32_, I32_, ctypes.POINTER(PlanOpts), ctypes.POINTER(P)],
        "ccl_execute": [P, ctypes.POINTER(P), ctypes.POINTER(P), P],
        "ccl_execute_host": [P, ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P), P],
        "ccl_execute_host_async": [P, ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P), P, P,
                                   P],
        "ccl_plan_status": [P],
        "ccl_plan_stats": [P, ctypes.POINTER(PlanStats)],
        "ccl_plan_timeline": [P, ctypes.POINTER(ctypes.c_double), I32_, ctypes.POINTER(ctypes.c_double),
                              ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)],
        "ccl_plan_timeline_raw": [P, ctypes.POINTER(ctypes.c_uint64), I64_, ctypes.POINTER(ctypes.c_int32), I32_,
                                  ctypes.POINTER(ctypes.c_int64)],
        "ccl_plan_steps": [P, ctypes.POINTER(StepInfo), I64_, ctypes.POINTER(ctypes.c_int64)],
        "ccl_plan_debug_drop_signal": [P, I32_, I32_],
        "ccl_plan_check": [P, I64_, I32_, ctypes.POINTER(PlanOpts), ctypes.POINTER(PlanStats)],
        "ccl_schedule_timeline": [P, I32_, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)],
        "ccl_allreduce_ring_noalloc": [ctypes.POINTER(P), ctypes.POINTER(P), I32_, I64_, I32_, I32_, P],
        "ccl_tune": [P, I64_, I32_, ctypes.POINTER(P), ctypes.POINTER(P), P, ctypes.POINTER(TuneOpts),
                     ctypes.POINTER(PlanOpts), ctypes.POINTER(PlanOpts), ctypes.POINTER(TuneReport)],
        "ccl_tune_table": [P, I32_, ctypes.POINTER(ctypes.c_int64), I32_, ctypes.POINTER(P), ctypes.POINTER(P), P,
                           ctypes.POINTER(TuneOpts), ctypes.POINTER(PlanOpts), ctypes.POINTER(TuneRow)],
        "ccl_tune_table_write_json": [ctypes.POINTER(TuneRow), I32_, I32_, ctypes.c_char_p, ctypes.c_char_p],
        "ccl_tune_table_read_json": [ctypes.c_char_p, ctypes.POINTER(TuneRow), I32_, ctypes.POINTER(ctypes.c_int32),
                                     ctypes.POINTER(ctypes.c_int32)],
        "ccl_tune_table_lookup": [ctypes.POINTER(TuneRow), I32_, I64_, ctypes.POINTER(PlanOpts)],
        "ccl_schedule_write_json": [P, ctypes.c_char_p],
        "ccl_plan_codegen_source": [P, I64_, I32_, ctypes.POINTER(PlanOpts), ctypes.c_char_p, ctypes.c_size_t,
                                    ctypes.POINTER(ctypes.c_size_t), I32_, ctypes.POINTER(ctypes.c_int64)],
        "ccl_schedule_read_json": [ctypes.c_char_p, ctypes.POINTER(P)],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    L.ccl_schedule_destroy.argtypes = [P]
    L.ccl_schedule_destroy.restype = None
    L.ccl_plan_destroy.argtypes = [P]
    L.ccl_plan_destroy.restype = None
    L.ccl_plan_opts_default.argtypes = [ctypes.POINTER(PlanOpts)]
    L.ccl_plan_opts_default.restype = None
    for name in ("ccl_last_error_detail", "ccl_version"):
        getattr(L, name).restype = ctypes.c_char_p
        getattr(L, name).argtypes = []
    L.ccl_tune_search.restype = ctypes.c_int
    L.ccl_tune_search.argtypes = [ctypes.POINTER(PlanOpts), ctypes.POINTER(TuneOpts), PROBE_FN, P,
                                  ctypes.POINTER(PlanOpts), ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_int32)]
    L.ccl_error_string.restype = ctypes.c_char_p
    L.ccl_error_string.argtypes = [ctypes.c_int]
    return L


lib = _load()
LIB_PATH = _LIB_PATH


def _check(code):
    if code != 0:
        raise CclError(code, lib.ccl_last_error_detail().decode())


def _ptrs(bufs):
    """Device (or host) addresses of a list of torch tensors / ints."""
    arr = (ctypes.c_void_p * len(bufs))()
    for i, b in enumerate(bufs):
        arr[i] = b if isinstance(b, int) else b.data_ptr()
    return arr


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def default_opts() -> PlanOpts:
    o = PlanOpts()
    lib.ccl_plan_opts_default(ctypes.byref(o))
    return o


_OPT_NAMES = frozenset(f[0] for f in PlanOpts._fields_)


def _with_opts(opts, kw) -> PlanOpts:
    """Library defaults (or ``opts``) with keyword overrides; an unknown
    keyword is an error rather than a silently ignored attribute."""
    o = opts if opts is not None else default_opts()
    for k, v in kw.items():
        if k not in _OPT_NAMES:
            raise TypeError(f"unknown plan option {k!r}")
        setattr(o, k, v)
    return o


class Schedule:
    """A compiled chunk program (``ccl_schedule_t``)."""

    def __init__(self, handle):
        self._h = ctypes.c_void_p(handle)

    @classmethod
    def builtin(cls, kind, nranks, group_size=0, flags=0):
        h = ctypes.c_void_p()
        _check(lib.ccl_schedule_builtin(kind, nranks, group_size, flags, ctypes.byref(h)))
        return cls(h.value)

    @classmethod
    def alltoallv(cls, counts, flags=0):
        """Uneven AllToAll: ``counts[s][d]`` chunks from rank s to rank d
        (``ccl_schedule_alltoallv``)."""
        rows = [[int(c) for c in row] for row in counts]
        R = len(rows)
        if any(len(r) != R for r in rows):
            raise ValueError("counts must be square")
        arr = (ctypes.c_int32 * max(1, R * R))(*[c for r in rows for c in r])
        h = ctypes.c_void_p()
        _check(lib.ccl_schedule_alltoallv(R, arr, flags, ctypes.byref(h)))
        return cls(h.value)

    @classmethod
    def compile(cls, ops, nranks, nchunks, fuse=True):
        """``ops``: iterable of 8-int rows (op, src_rank, src_buf, src_off,
        dst_rank, dst_buf, dst_off, count).  ``fuse``: a bool, or one of
        FUSE_NONE / FUSE_FULL / FUSE_NOCHAIN."""
        rows = [tuple(int(v) for v in r) for r in ops]
        arr = (Op * max(1, len(rows)))(*[Op(*r) for r in rows])
        nch = (ctypes.c_int32 * 3)(*[int(c) for c in nchunks])
        h = ctypes.c_void_p()
        mode = int(fuse) if not isinstance(fuse, bool) else (FUSE_FULL if fuse else FUSE_NONE)
        _check(lib.ccl_schedule_compile(arr, len(rows), nranks, nch, mode, ctypes.byref(h)))
        return cls(h.value)

    def info(self) -> ScheduleInfo:
        i = ScheduleInfo()
        _check(lib.ccl_schedule_info(self._h, ctypes.byref(i)))
        return i

    def ops(self):
        n = ctypes.c_int32()
        lib.ccl_schedule_get_ops(self._h, None, 0, ctypes.byref(n))
        arr = (Op * max(1, n.value))()
        _check(lib.ccl_schedule_get_ops(self._h, arr, n.value, ctypes.byref(n)))
        return [tuple(getattr(arr[i], f) for f, _ in Op._fields_) for i in range(n.value)]

    def instrs(self):
        n = ctypes.c_int32()
        lib.ccl_schedule_get_instrs(self._h, None, 0, ctypes.byref(n))
        arr = (InstrInfo * max(1, n.value))()
        _check(lib.ccl_schedule_get_instrs(self._h, arr, n.value, ctypes.byref(n)))
        return [{f: getattr(arr[i], f) for f, _ in InstrInfo._fields_} for i in range(n.value)]

    def timeline(self, scheduler=SCHED_HPDS):
        """Sub-pipeline index of every transfer, and the sub-pipeline count."""
        n = self.info().ntransfers
        arr = (ctypes.c_int32 * max(1, n))()
        nsub = ctypes.c_int32()
        _check(lib.ccl_schedule_timeline(self._h, scheduler, arr, ctypes.byref(nsub)))
        return list(arr[:n]), nsub.value

    def save(self, path):
        """Write the schedule as JSON (``ccl_schedule_write_json``)."""
        _check(lib.ccl_schedule_write_json(self._h, os.fsencode(path)))

    @classmethod
    def load(cls, path):
        """Read a schedule written by ``save`` (``ccl_schedule_read_json``)."""
        h = ctypes.c_void_p()
        _check(lib.ccl_schedule_read_json(os.fsencode(path), ctypes.byref(h)))
        return cls(h.value)

    def codegen_source(self, chunk_elems, dtype, compile=False, opts: PlanOpts | None = None, **kw):
        """(source, cubin bytes or None) of the kernel a plan with codegen = 1
        would run (``ccl_plan_codegen_source``; host only)."""
        o = _with_opts(opts, kw)
        n = ctypes.c_size_t()
        cb = ctypes.c_int64()
        _check(lib.ccl_plan_codegen_source(self._h, chunk_elems, dtype, ctypes.byref(o), None, 0, ctypes.byref(n),
                                           0, None))
        buf = ctypes.create_string_buffer(n.value + 1)
        _check(lib.ccl_plan_codegen_source(self._h, chunk_elems, dtype, ctypes.byref(o), buf, n.value + 1,
                                           ctypes.byref(n), int(bool(compile)), ctypes.byref(cb)))
        return buf.value.decode(), (cb.value if compile else None)

    def check(self, chunk_elems, dtype, opts: PlanOpts | None = None, **kw) -> PlanStats:
        """Plan on the host only (deadlock simulation included, no GPU)."""
        o = _with_opts(opts, kw)
        st = PlanStats()
        _check(lib.ccl_plan_check(self._h, chunk_elems, dtype, ctypes.byref(o), ctypes.byref(st)))
        return st

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            lib.ccl_schedule_destroy(h)
            self._h = ctypes.c_void_p()


class Plan:
    """An executable plan (``ccl_plan_t``) on the current CUDA device."""

    def __init__(self, schedule: Schedule, chunk_elems: int, dtype: int, opts: PlanOpts | None = None, **kw):
        o = _with_opts(opts, kw)
        self.schedule = schedule
        self.opts = o
        self.dtype = dtype
        self.chunk_elems = chunk_elems
        h = ctypes.c_void_p()
        _check(lib.ccl_plan_create(schedule._h, chunk_elems, dtype, 0, ctypes.byref(o), ctypes.byref(h)))
        self._h = h
        info = schedule.info()
        self.nranks = info.nranks
        self.nchunks = tuple(info.nchunks)
        self.in_elems = info.nchunks[0] * chunk_elems
        self.out_elems = info.nchunks[1] * chunk_elems

    def execute(self, inputs, outputs, stream=None):
        _check(lib.ccl_execute(self._h, _ptrs(inputs), _ptrs(outputs), _stream(stream)))

    def execute_host_async(self, host_in, host_out, dev_in, dev_out, copy_in_stream, compute_stream,
                           copy_out_stream):
        """Input copies, kernel and output copies on three streams
        (``ccl_execute_host_async``)."""
        _check(lib.ccl_execute_host_async(self._h, _ptrs(host_in), _ptrs(host_out), _ptrs(dev_in), _ptrs(dev_out),
                                          _stream(copy_in_stream), _stream(compute_stream),
                                          _stream(copy_out_stream)))

    def execute_host(self, host_in, host_out, dev_in, dev_out, stream=None):
        _check(lib.ccl_execute_host(self._h, _ptrs(host_in), _ptrs(host_out), _ptrs(dev_in), _ptrs(dev_out),
                                    _stream(stream)))

    def status(self):
        _check(lib.ccl_plan_status(self._h))

    def stats(self) -> PlanStats:
        st = PlanStats()
        _check(lib.ccl_plan_stats(self._h, ctypes.byref(st)))
        return st

    def timeline(self):
        st = self.stats()
        idle = (ctypes.c_double * st.nthreadblocks)()
        mean, mx, span = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
        _check(lib.ccl_plan_timeline(self._h, idle, st.nthreadblocks, ctypes.byref(mean), ctypes.byref(mx),
                                     ctypes.byref(span)))
        return {"idle": list(idle), "mean_idle": mean.value, "max_idle": mx.value, "span_us": span.value}

    def timeline_raw(self):
        """(start, waited, first tile handed out, last tile done, posted) in ns
        per step as an (nsteps, 5) uint64 array, and the first step of every
        threadblock (ntb + 1 entries)."""
        import numpy as np
        st = self.stats()
        n = ctypes.c_int64()
        tb = (ctypes.c_int32 * (st.nthreadblocks + 1))()
        _check(lib.ccl_plan_timeline_raw(self._h, None, 0, tb, st.nthreadblocks + 1, ctypes.byref(n)))
        buf = np.zeros(5 * n.value, dtype=np.uint64)
        _check(lib.ccl_plan_timeline_raw(self._h, buf.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), buf.size, tb,
                                         st.nthreadblocks + 1, None))
        return buf.reshape(-1, 5), list(tb)

    def steps(self):
        """Every step of the plan in threadblock-program order, as dicts."""
        n = ctypes.c_int64()
        _check(lib.ccl_plan_steps(self._h, None, 0, ctypes.byref(n)))
        arr = (StepInfo * max(1, n.value))()
        _check(lib.ccl_plan_steps(self._h, arr, n.value, ctypes.byref(n)))
        return [{f: getattr(s, f) for f, _ in StepInfo._fields_} for s in arr[:n.value]]

    def debug_drop_signal(self, tb, step):
        _check(lib.ccl_plan_debug_drop_signal(self._h, tb, step))

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            lib.ccl_plan_destroy(h)
            self._h = ctypes.c_void_p()


def tune(schedule: Schedule, chunk_elems, dtype, inputs, outputs, stream=None, start: PlanOpts | None = None,
         max_rounds=3, reps=5, min_gain=0.01, max_channels=0):
    best = PlanOpts()
    rep = TuneReport()
    to = TuneOpts(max_rounds, reps, min_gain, max_channels)
    _check(lib.ccl_tune(schedule._h, chunk_elems, dtype, _ptrs(inputs), _ptrs(outputs), _stream(stream),
                        ctypes.byref(to), ctypes.byref(start) if start is not None else None, ctypes.byref(best),
                        ctypes.byref(rep)))
    return best, rep


def tune_table(schedule: Schedule, dtype, sizes, inputs, outputs, stream=None, start: PlanOpts | None = None,
               max_rounds=3, reps=5, min_gain=0.01, max_channels=0):
    """Per-size tuning (``ccl_tune_table``): a list of TuneRow, one per
    chunk size in ``sizes``; the buffers hold the largest size."""
    n = len(sizes)
    arr = (ctypes.c_int64 * n)(*[int(x) for x in sizes])
    rows = (TuneRow * n)()
    to = TuneOpts(max_rounds, reps, min_gain, max_channels)
    _check(lib.ccl_tune_table(schedule._h, dtype, arr, n, _ptrs(inputs), _ptrs(outputs), _stream(stream),
                              ctypes.byref(to), ctypes.byref(start) if start is not None else None, rows))
    return list(rows)


def write_tune_table(rows, dtype, path, note=""):
    arr = (TuneRow * max(1, len(rows)))(*rows)
    _check(lib.ccl_tune_table_write_json(arr, len(rows), dtype, note.encode(), os.fsencode(path)))


def read_tune_table(path):
    """(rows, dtype) of a table file."""
    n, dt = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.ccl_tune_table_read_json(os.fsencode(path), None, 0, ctypes.byref(n), ctypes.byref(dt)))
    rows = (TuneRow * max(1, n.value))()
    _check(lib.ccl_tune_table_read_json(os.fsencode(path), rows, n.value, ctypes.byref(n), ctypes.byref(dt)))
    return list(rows[:n.value]), dt.value


def lookup_tune_table(rows, chunk_elems) -> PlanOpts:
    arr = (TuneRow * max(1, len(rows)))(*rows)
    o = PlanOpts()
    _check(lib.ccl_tune_table_lookup(arr, len(rows), chunk_elems, ctypes.byref(o)))
    return o


def allreduce_ring_noalloc(inputs, outputs, chunk_elems, dtype, channels=0, stream=None):
    """Ring AllReduce with no device allocation (static scratch; see ccl.h)."""
    _check(lib.ccl_allreduce_ring_noalloc(_ptrs(inputs), _ptrs(outputs), len(inputs), chunk_elems, dtype,
                                          channels, _stream(stream)))


def tune_search(probe, start: PlanOpts | None = None, max_rounds=3, min_gain=0.01):
    """Run the tuner's search with a Python probe(opts) -> bandwidth."""
    cb = PROBE_FN(lambda user, o: float(probe(o.contents)))
    best = PlanOpts()
    bw = ctypes.c_double()
    n = ctypes.c_int32()
    to = TuneOpts(max_rounds, 1, min_gain, 0)
    _check(lib.ccl_tune_search(ctypes.byref(start) if start is not None else None, ctypes.byref(to), cb, None,
                               ctypes.byref(best), ctypes.byref(bw), ctypes.byref(n)))
    return best, bw.value, n.value


def version() -> str:
    return lib.ccl_version().decode()
