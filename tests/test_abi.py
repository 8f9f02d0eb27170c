"""The C ABI library loads and exports every function include/ccl.h declares
(no GPU needed: nothing here launches work)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_\s\*]*?\b(ccl_[A-Za-z0-9_]+)\s*\(", text, re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("ccl_schedule_compile", "ccl_schedule_builtin", "ccl_plan_create", "ccl_execute",
                 "ccl_execute_host", "ccl_plan_status", "ccl_plan_stats", "ccl_tune", "ccl_plan_destroy",
                 "ccl_schedule_destroy", "ccl_error_string", "ccl_last_error_detail"):
        assert must in names, must


def test_library_exports_every_declared_symbol():
    import collective_communication_schedule_gb300 as ccl
    lib = ctypes.CDLL(ccl.LIB_PATH)
    missing = [n for n in sorted(declared_functions()) if not hasattr(lib, n)]
    assert not missing, missing


def test_host_only_calls_work_without_a_gpu():
    import collective_communication_schedule_gb300 as ccl
    assert "sm_103a" in ccl.version()
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 8)
    assert s.info().nranks == 8
    st = s.check(1024, ccl.F32, channels=2)
    assert st.nthreadblocks == 16
    assert ccl.lib.ccl_error_string(3) == b"deadlock"


def test_binding_structs_match_the_header_layout(tmp_path):
    """Every ctypes structure of the binding has the size and field offsets of
    its C counterpart, as gcc lays it out from include/ccl.h."""
    import shutil
    import subprocess
    import pytest
    import collective_communication_schedule_gb300 as ccl
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    pairs = [(ccl.Op, "ccl_op_t"), (ccl.ScheduleInfo, "ccl_schedule_info_t"), (ccl.InstrInfo, "ccl_instr_info_t"),
             (ccl.PlanOpts, "ccl_plan_opts_t"), (ccl.PlanStats, "ccl_plan_stats_t"), (ccl.StepInfo, "ccl_step_info_t"),
             (ccl.TuneOpts, "ccl_tune_opts_t"), (ccl.TuneReport, "ccl_tune_report_t"), (ccl.TuneRow, "ccl_tune_row_t")]
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "ccl.h"', "int main(void) {"]
    want = []
    for cls, cname in pairs:
        lines.append(f'    printf("%zu\\n", sizeof({cname}));')
        want.append(ctypes.sizeof(cls))
        for f in cls._fields_:
            lines.append(f'    printf("%zu\\n", offsetof({cname}, {f[0]}));')
            want.append(getattr(cls, f[0]).offset)
    lines += ["    return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    assert got == want


def test_binding_constants_match_the_header():
    """Every CCL_* constant of the header that the binding re-exports (same
    name without the prefix) has the header's value."""
    import collective_communication_schedule_gb300 as ccl
    vals = {}
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", fn)).read(), flags=re.S)
        for m in re.finditer(r"#define\s+CCL_([A-Z0-9_]+)\s+(\d+)u?\b", text):
            vals[m.group(1)] = int(m.group(2))
        for m in re.finditer(r"\bCCL_([A-Z0-9_]+)\s*=\s*(-?\d+)", text):
            vals[m.group(1)] = int(m.group(2))
    checked = 0
    for name, v in vals.items():
        if hasattr(ccl, name) and isinstance(getattr(ccl, name), int):
            assert getattr(ccl, name) == v, name
            checked += 1
    assert checked >= 20
    # instruction kind names are indexed by the header's CCL_I_* values
    for i, name in enumerate(ccl.KIND_NAMES):
        assert vals["I_" + name.upper()] == i, name
    # the compiler's kinds, then the kinds only plans contain (direct
    # transport's folds)
    plan_only = ["copy2", "rrc2", "rrs3", "rrc3", "rrcs3", "rsend", "rcsend", "rrc3d", "reduce2", "copy3"]
    assert vals["I_NKINDS"] == len(ccl.KIND_NAMES) - len(plan_only) and ccl.KIND_NAMES[vals["I_NKINDS"]:] == plan_only


def test_layout_header_codes_match_the_c_abi():
    """The codes the run-time-compiled kernels take from the layout header
    (which cannot include the C ABI header) have the C ABI's values."""
    def codes(path):
        text = re.sub(r"/\*.*?\*/|//[^\n]*", "", open(path).read(), flags=re.S)
        vals = {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(CCL_[A-Z0-9_]+)\s*=\s*(-?\d+)", text)}
        for m in re.finditer(r"#define\s+(CCL_[A-Z0-9_]+)\s+(\d+)\b", text):
            vals[m.group(1)] = int(m.group(2))
        return vals
    abi = codes(os.path.join(ROOT, "include", "ccl.h"))
    layout = codes(os.path.join(ROOT, "collective_communication_schedule_gb300", "csrc", "ccl_layout.h"))
    assert len(layout) >= 18
    for name, v in layout.items():
        assert abi.get(name) == v, name


def test_default_options_set_every_field():
    """ccl_plan_opts_default writes every field of ccl_plan_opts_t: the
    result does not depend on what the memory held before."""
    import collective_communication_schedule_gb300 as ccl
    a = ccl.PlanOpts.from_buffer_copy(b"\x5a" * ctypes.sizeof(ccl.PlanOpts))
    b = ccl.PlanOpts.from_buffer_copy(b"\x00" * ctypes.sizeof(ccl.PlanOpts))
    ccl.lib.ccl_plan_opts_default(ctypes.byref(a))
    ccl.lib.ccl_plan_opts_default(ctypes.byref(b))
    for f, _ in ccl.PlanOpts._fields_:
        assert getattr(a, f) == getattr(b, f), f
