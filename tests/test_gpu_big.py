"""Whole-model streamed workloads at full size (configs 4 and 5), each in a child
process so that its pinned host state is released when it ends."""
import gc
import json
import os
import subprocess
import sys

import pytest

from gpu_common import ensure_library

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_library()


@pytest.mark.parametrize("cid", [4, 5])
def test_whole_model_streamed_full_size(cid):
    import oracle_cache
    oracle_cache._cache.clear()
    gc.collect()
    r = subprocess.run([sys.executable, os.path.join(HERE, "big_config_check.py"), str(cid)],
                       capture_output=True, text=True, timeout=3000)
    tail = (r.stdout.strip().splitlines() or [""])[-1]
    if r.returncode == 3:
        pytest.skip(f"not enough host memory for config {cid}: {tail}")
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    res = json.loads(tail)
    assert res["tensors_checked"] == res["tensors"] and res["params_checked"] == res["params"]
    assert res["non_bit_exact"] == 0
