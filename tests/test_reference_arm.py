"""The benchmark's reference arm (the oracle on the host cores) runs without
the product: no module of the CUDA library's package is imported and no
library of it is loaded."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_uses_only_the_oracle():
    code = (
        "import sys, json, types\n"
        "sys.argv = ['bench.py', '--impl', 'reference', '--steps', '1', '--warmup', '0', '--only', 'ar_1m,ag_3m']\n"
        "import bench\n"
        "bench.main()\n"
        "assert not any(m.startswith('collective_communication_schedule_gb300') for m in sys.modules), 'package imported'\n"
        "maps = open('/proc/self/maps').read()\n"
        "assert 'libccl' not in maps, 'libccl loaded'\n"
        "assert 'liboracle' in maps\n"
    )
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    import json
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
