"""The checked build and the device-side input checks.

- libdflash_checked.so (DFLASH_CHECKED) carries device bounds assertions on
  the addresses the kernels compute; a failed one reports DFLASH_ERR_CHECK
  through the status word instead of trapping.  The small parity tests (and
  the streaming-attention comparisons) run against it in a child process:
  every result must still match and every status word must stay clean.
- Token ids read on the device are checked in every build: an out-of-range
  anchor comes back as DFLASH_ERR_INVALID_ARG (its row reads token 0, no
  access leaves the table), and the next clean call as DFLASH_OK.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from block_diffusion_speculative_step_gb300 import dflash as D
from tests import gpu_common as G
from tests import helpers as Hh

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_suite_on_the_checked_build():
    env = dict(os.environ, DFLASH_LIB="checked")
    sel = "causal_layer or bidir_layer or draft_block or verify_accept or fuse_context or lossless or rows_independent"
    code = ("import sys\n"
            f"sys.path.insert(0, {ROOT!r})\n"
            "from block_diffusion_speculative_step_gb300 import dflash as D\n"
            "assert D.dflash_build_flags() == D.DFLASH_BUILD_CHECKED, 'not the checked library'\n"
            "import pytest\n"
            f"sys.exit(pytest.main(['-q', '-p', 'no:cacheprovider', '-m', 'gpu', "
            f"{os.path.join(ROOT, 'tests', 'test_gpu_parity.py')!r}, '-k', {sel!r}, "
            f"{os.path.join(ROOT, 'tests', 'test_gpu_paged.py')!r}, "
            f"{os.path.join(ROOT, 'tests', 'test_gpu_attn_stream.py')!r}]))\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout


def test_out_of_range_token_id_is_reported():
    assert D.dflash_build_flags() == 0  # this process runs the normal library
    w = Hh.small_workload("bf16", H=256, nq=4, nkv=2, d=64, I=384, V=1000, t_layers=1, d_layers=1,
                          taps=(0, 0), block=8)
    eng, om, _ = G.setup(w, S=2, cap=64)
    eng.base_pos.fill_(10)
    eng.anchor.copy_(torch.tensor([5, w.vocab + 7], dtype=torch.int32))
    eng.draft()
    assert eng.status() == D.DFLASH_ERR_INVALID_ARG
    assert "status word" in D.dflash_last_error()
    eng.anchor.copy_(torch.tensor([5, 6], dtype=torch.int32))
    eng.draft()
    assert eng.status() == D.DFLASH_OK
