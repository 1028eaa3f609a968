"""The mma.sync cluster attention for head dimension 128 (opt-in with
DFLASH_ATTN_MMASYNC=1; the default there is the tcgen05 kernel): the same
attention parity tests, run in a child process with the switch set --
S = QK^T and O += PV as mma.sync m16n8k16 tiles, key quarters merged in
shared memory, ranks through distributed shared memory."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_attention_parity_with_mmasync_kernel():
    env = dict(os.environ, DFLASH_ATTN_MMASYNC="1")
    sel = "long_context or causal_layer or bidir_layer or draft_block or rows_independent or lossless"
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "gpu",
                        os.path.join(ROOT, "tests", "test_gpu_parity.py"), "-k", sel,
                        os.path.join(ROOT, "tests", "test_gpu_fullsize.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
