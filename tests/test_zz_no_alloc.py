"""The allocation-free ring AllReduce entry point, called through the C ABI.

Some callers cannot allocate device memory when they run a collective (their
device memory is pre-reserved by a framework allocator, or a cudaMalloc's
possible device-wide synchronisation is not acceptable mid-step).
``ccl_allreduce_ring_noalloc`` serves them with scratch in a static device
array.  Its results must equal the plan path's bit for bit (same ring
reduction order), on two calls in a row because the array keeps the previous
call's contents.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

BF16, F32 = 1, 0


def _fn():
    import collective_communication_schedule_gb300 as ccl
    lib = ctypes.CDLL(ccl.LIB_PATH)
    f = lib.ccl_allreduce_ring_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32,
                  ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
    return ccl, lib, f


def _ptrs(ts):
    a = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        a[i] = t.data_ptr()
    return a


@pytest.mark.parametrize("dtype,ce,channels", [(BF16, 20003, 0), (F32, 65536, 4)])
def test_noalloc_equals_plan_path_on_two_calls(dtype, ce, channels):
    import torch
    import datagen
    ccl, lib, f = _fn()
    R = 8
    plan = ccl.Plan(ccl.Schedule.builtin(ccl.RING_ALLREDUCE, R), ce, dtype, channels=2)
    tdt = torch.int16 if dtype == BF16 else torch.float32
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        host = datagen.rank_inputs(60 + call, "normal", R, R * ce, dtype)
        ins = [torch.from_numpy(a.view(np.int16) if dtype == BF16 else a).cuda() for a in host]
        ref = [torch.empty(R * ce, dtype=tdt, device="cuda") for _ in range(R)]
        out = [torch.full((R * ce,), 7, dtype=tdt, device="cuda") for _ in range(R)]
        plan.execute(ins, ref)
        rc = f(_ptrs(ins), _ptrs(out), R, ce, dtype, channels, ctypes.c_void_p(stream))
        assert rc == 0, lib.ccl_last_error_detail and ctypes.c_char_p(lib.ccl_last_error_detail()).value
        torch.cuda.synchronize()
        plan.status()
        for r in range(R):
            assert torch.equal(out[r].view(torch.uint8), ref[r].view(torch.uint8)), f"call {call} rank {r}"


def test_noalloc_rejects_more_links_than_the_static_scratch_holds():
    import torch
    ccl, lib, f = _fn()
    R = 16
    bufs = [torch.empty(R * 64, dtype=torch.float32, device="cuda") for _ in range(R)]
    rc = f(_ptrs(bufs), _ptrs(bufs), R, 64, F32, 8, None)   # 16 x 8 = 128 links > 64
    assert rc == 1
    lib.ccl_last_error_detail.restype = ctypes.c_char_p
    assert b"exceeds" in lib.ccl_last_error_detail()
