"""Schedules and per-size tuning tables written to JSON files and read back
(host only: no GPU involved)."""
import json

import pytest

ccl = pytest.importorskip("collective_communication_schedule_gb300")

F32, BF16 = 0, 1


@pytest.mark.parametrize("kind,R,G,flags", [(0, 8, 0, 0), (3, 16, 8, 4), (4, 8, 4, 0), (5, 24, 8, 2), (1, 5, 0, 1)])
def test_schedule_round_trip(tmp_path, kind, R, G, flags):
    s = ccl.Schedule.builtin(kind, R, G, flags)
    path = tmp_path / "s.json"
    s.save(path)
    t = ccl.Schedule.load(path)
    assert t.ops() == s.ops() and t.instrs() == s.instrs()
    a, b = s.info(), t.info()
    assert (a.builtin, a.group_size, a.nranks, tuple(a.nchunks)) == (b.builtin, b.group_size, b.nranks, tuple(b.nchunks))
    sa, sb = s.check(1000, F32, channels=2), t.check(1000, F32, channels=2)
    assert (sa.schedule_bytes, sa.nsteps, sa.nthreadblocks, sa.busbw_factor) == \
        (sb.schedule_bytes, sb.nsteps, sb.nthreadblocks, sb.busbw_factor)


def test_user_program_round_trip_keeps_its_fusion_mode(tmp_path):
    ops = [(0, 0, 0, 0, 1, 1, 0, 1), (1, 1, 1, 0, 2, 1, 0, 1), (0, 2, 1, 0, 0, 1, 1, 1)]
    for fuse in (ccl.FUSE_NONE, ccl.FUSE_FULL, ccl.FUSE_NOCHAIN):
        s = ccl.Schedule.compile(ops, 3, (1, 2, 0), fuse=fuse)
        s.save(tmp_path / "p.json")
        t = ccl.Schedule.load(tmp_path / "p.json")
        assert t.instrs() == s.instrs()
        assert json.loads((tmp_path / "p.json").read_text())["fuse"] == fuse


def test_schedule_file_with_another_digest_or_bad_content_is_refused(tmp_path):
    s = ccl.Schedule.builtin(0, 4)
    p = tmp_path / "s.json"
    s.save(p)
    d = json.loads(p.read_text())
    d["instr_digest"] = "123"
    p.write_text(json.dumps(d))
    with pytest.raises(ccl.CclError) as e:
        ccl.Schedule.load(p)
    assert e.value.code == 1 and "other instructions" in e.value.detail
    p.write_text("{\"format\": \"ccl-schedule-1\", \"nranks\": 4,")
    with pytest.raises(ccl.CclError):
        ccl.Schedule.load(p)
    with pytest.raises(ccl.CclError):
        ccl.Schedule.load(tmp_path / "missing.json")
    d = json.loads(json.dumps({"format": "other"}))
    p.write_text(json.dumps(d))
    with pytest.raises(ccl.CclError):
        ccl.Schedule.load(p)


def _row(ce, channels, nthreads, slot, engine, us):
    r = ccl.TuneRow()
    r.chunk_elems = ce
    r.best = ccl.default_opts()
    r.best.channels, r.best.nthreads, r.best.slot_bytes, r.best.engine = channels, nthreads, slot, engine
    r.report.probes, r.report.best_us, r.report.default_us, r.report.best_gbs = 17, us, 2 * us, 1.5
    return r


def test_tune_table_round_trip_and_lookup(tmp_path):
    rows = [_row(2048, 1, 512, 16384, 1, 20.5), _row(16384, 2, 512, 131072, 1, 31.25),
            _row(196608, 4, 1024, 131072, 0, 80.0)]
    p = tmp_path / "t.json"
    ccl.write_tune_table(rows, BF16, p, note="ring AllGather R=8")
    back, dt = ccl.read_tune_table(p)
    assert dt == BF16 and len(back) == 3
    for a, b in zip(rows, back):
        assert a.chunk_elems == b.chunk_elems
        for f, _ in ccl.PlanOpts._fields_:
            assert getattr(a.best, f) == getattr(b.best, f), f
        assert (a.report.probes, a.report.best_us, a.report.default_us) == \
            (b.report.probes, b.report.best_us, b.report.default_us)
    assert json.loads(p.read_text())["note"] == "ring AllGather R=8"
    # nearest size on a log scale
    assert ccl.lookup_tune_table(back, 2048).channels == 1
    assert ccl.lookup_tune_table(back, 4096).channels == 1       # 2x from 2048, 4x from 16384
    assert ccl.lookup_tune_table(back, 8192).channels == 2       # 4x vs 2x
    assert ccl.lookup_tune_table(back, 1 << 20).channels == 4
    assert ccl.lookup_tune_table(back, 1).channels == 1


def test_tune_table_missing_fields_take_defaults(tmp_path):
    p = tmp_path / "t.json"
    p.write_text(json.dumps({"format": "ccl-tune-table-1", "dtype": 0,
                             "rows": [{"chunk_elems": 64, "opts": {"channels": 3}}]}))
    rows, dt = ccl.read_tune_table(p)
    d = ccl.default_opts()
    assert rows[0].best.channels == 3 and rows[0].best.slot_bytes == d.slot_bytes and dt == 0
    p.write_text(json.dumps({"format": "ccl-tune-table-1", "dtype": 0, "rows": [{"opts": {}}]}))
    with pytest.raises(ccl.CclError):
        ccl.read_tune_table(p)


def test_search_respects_the_channel_limit():
    """A surface that grows with channels: the search stops at the limit."""
    def probe(o):
        return float(o.channels) + 0.001 * o.nthreads
    best, bw, n = ccl.tune_search(probe)
    assert best.channels == 48
    to = ccl.TuneOpts(3, 1, 0.01, 4)
    b = ccl.PlanOpts()
    bwv = ccl.ctypes.c_double()
    nn = ccl.ctypes.c_int32()
    cb = ccl.PROBE_FN(lambda user, o: float(probe(o.contents)))
    assert ccl.lib.ccl_tune_search(None, ccl.ctypes.byref(to), cb, None, ccl.ctypes.byref(b), ccl.ctypes.byref(bwv),
                                   ccl.ctypes.byref(nn)) == 0
    assert b.channels == 4
