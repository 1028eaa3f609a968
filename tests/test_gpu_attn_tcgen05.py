"""The tcgen05 attention kernel (opt-in with DFLASH_ATTN_TCGEN05=1): the
same attention parity tests, run in a child process with the switch set --
S = QK^T and O += PV on the 5th-generation tensor cores with TMEM
accumulators, the softmax shared by four warps over duplicated score rows."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_attention_parity_with_tcgen05_kernel():
    env = dict(os.environ, DFLASH_ATTN_TCGEN05="1")
    sel = "long_context or causal_layer or bidir_layer or draft_block or rows_independent or lossless"
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "gpu",
                        os.path.join(ROOT, "tests", "test_gpu_parity.py"), "-k", sel,
                        os.path.join(ROOT, "tests", "test_gpu_fullsize.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
