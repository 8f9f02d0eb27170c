"""The allocation-free ring AllReduce entry point, called through the C ABI.

Some callers cannot allocate device memory when they run a collective: their
device memory is pre-reserved by a framework allocator, or a cudaMalloc's
possible device-wide synchronisation is not acceptable in the middle of a
step.  ``ccl_allreduce_ring_noalloc`` serves them with its scratch in a static
device array.  Its results must equal, bit for bit, both the plan path's
(same ring reduction order) and the oracle's, on two calls in a row because
the array keeps the previous call's contents.  Also covered: one rank (a
plain copy), chunks smaller than one vector per channel (empty pieces that
still pass their flags on), and in-place calls.  This file is collected last
on purpose.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

F32, BF16, I32 = 0, 1, 3
TORCH_DT = {F32: "float32", BF16: "int16", I32: "int32"}
DIST = {F32: "normal", BF16: "normal", I32: "int"}


def _fn():
    import collective_communication_schedule_gb300 as ccl
    lib = ctypes.CDLL(ccl.LIB_PATH)
    f = lib.ccl_allreduce_ring_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32,
                  ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
    lib.ccl_last_error_detail.restype = ctypes.c_char_p
    lib.ccl_last_error_detail.argtypes = []
    return ccl, lib, f


def _ptrs(ts):
    a = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        a[i] = t.data_ptr()
    return a


def _host(t, dtype):
    a = t.cpu().numpy()
    return a.view(np.uint16) if dtype == BF16 else a


@pytest.mark.parametrize("R,dtype,ce,channels,inplace", [
    (8, BF16, 20003, 0, False),   # ragged chunk, default channels
    (8, F32, 65536, 4, False),    # several slots and micro-batches per channel
    (8, I32, 4099, 2, False),
    (1, F32, 1000, 0, False),     # one rank: a copy
    (8, F32, 3, 8, False),        # 3 elements over 8 channels: empty pieces
    (5, BF16, 7777, 3, True),     # in place
    (8, F32, 40000, 0, True),
])
def test_noalloc_equals_oracle_and_plan_path_on_two_calls(R, dtype, ce, channels, inplace):
    import torch
    import datagen
    import oracle
    from oracle import schedules as OS
    ccl, lib, f = _fn()
    tdt = getattr(torch, TORCH_DT[dtype])
    plan = ccl.Plan(ccl.Schedule.builtin(ccl.RING_ALLREDUCE, R), ce, dtype, channels=2)
    ops, nch = OS.ring_allreduce(R)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        host = datagen.rank_inputs(60 + call, DIST[dtype], R, R * ce, dtype)
        dev = [torch.from_numpy(a.view(np.int16) if dtype == BF16 else a).cuda() for a in host]
        ref = [torch.empty(R * ce, dtype=tdt, device="cuda") for _ in range(R)]
        plan.execute(dev, ref)
        if inplace:
            ins = outs = [t.clone() for t in dev]
        else:
            ins = dev
            outs = [torch.full((R * ce,), 7, dtype=tdt, device="cuda") for _ in range(R)]
        rc = f(_ptrs(ins), _ptrs(outs), R, ce, dtype, channels, ctypes.c_void_p(stream))
        assert rc == 0, lib.ccl_last_error_detail()
        torch.cuda.synchronize()
        plan.status()
        want, _, _ = oracle.run(ops, R, nch, ce, dtype, host)
        for r in range(R):
            got = _host(outs[r], dtype)
            assert np.array_equal(got.view(np.uint8), want[r].view(np.uint8)), f"call {call} rank {r} vs oracle"
            assert torch.equal(outs[r].view(torch.uint8), ref[r].view(torch.uint8)), f"call {call} rank {r} vs plan"


def test_noalloc_rejects_more_links_than_the_static_scratch_holds():
    import torch
    ccl, lib, f = _fn()
    R = 16
    bufs = [torch.empty(R * 64, dtype=torch.float32, device="cuda") for _ in range(R)]
    rc = f(_ptrs(bufs), _ptrs(bufs), R, 64, F32, 8, None)   # 16 x 8 = 128 links > 64
    assert rc == 1
    assert b"exceeds" in lib.ccl_last_error_detail()
