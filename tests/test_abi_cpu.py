"""The C-ABI library without a GPU: it builds, loads, exports every function
include/dflash.h declares, its ctypes mirrors match the C struct layouts, and
host-side argument checks fail cleanly before any launch."""
import ctypes as C
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


@pytest.fixture(scope="module")
def D():
    from block_diffusion_speculative_step_gb300 import build
    build.build()
    import torch  # noqa: F401  (loads the shared CUDA runtime first, as in use)
    from block_diffusion_speculative_step_gb300 import dflash
    return dflash


def header_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(dflash_\w+)\s*\(", src, re.M)))


def test_exports_match_header(D):
    declared = header_functions()
    assert set(declared) == set(D.EXPORTS), (declared, D.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", D._build.LIB], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    for name in declared:
        assert name in exported, name
        getattr(D.lib(), name)


def test_abi_version(D):
    v = int(re.search(r"#define DFLASH_ABI_VERSION (\d+)", open(HEADER).read()).group(1))
    assert D.dflash_abi_version() == v


def test_struct_layouts_match_c(D):
    structs = ["dflash_dims", "dflash_kv", "dflash_layer_weights", "dflash_embed_args", "dflash_layer_args",
               "dflash_fuse_args", "dflash_draft_args", "dflash_verify_args", "dflash_path_args",
               "dflash_sample_drafts_args", "dflash_sample_accept_args", "dflash_trace_stat"]
    lines = ["#include <stdio.h>", "#include <stddef.h>", f'#include "{HEADER}"', "int main(void) {"]
    for s in structs:
        lines.append(f'  printf("{s} %zu\\n", sizeof({s}));')
        for fname, _ in getattr(D, s)._fields_:
            lines.append(f'  printf("{s}.{fname} %zu\\n", offsetof({s}, {fname}));')
    lines.append("  return 0; }")
    with tempfile.TemporaryDirectory() as td:
        src = os.path.join(td, "l.c")
        exe = os.path.join(td, "l")
        open(src, "w").write("\n".join(lines))
        subprocess.check_call(["gcc", "-o", exe, src])
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    ref = dict(l.rsplit(" ", 1) for l in out.splitlines())
    for s in structs:
        cls = getattr(D, s)
        assert C.sizeof(cls) == int(ref[s]), s
        for fname, _ in cls._fields_:
            assert getattr(cls, fname).offset == int(ref[f"{s}.{fname}"]), f"{s}.{fname}"


def test_invalid_arguments_fail_before_launch(D):
    L = D.lib()
    # NULL argument structs
    for name in ("dflash_embed", "dflash_decoder_layer_forward", "dflash_fuse_context", "dflash_draft_block",
                 "dflash_verify_accept", "dflash_path_select", "dflash_sample_drafts", "dflash_sample_accept"):
        assert getattr(L, name)(None, None, 0, None) == D.DFLASH_ERR_INVALID_ARG
        assert "NULL args" in D.dflash_last_error()
    # bad dims
    a = D.dflash_embed_args()
    a.dims = D.dflash_dims(256, 4, 3, 64, 512, 1000, 1e4, 1e-6, D.DFLASH_BF16)  # 4 % 3 != 0
    assert L.dflash_embed(C.byref(a), None, 0, None) == D.DFLASH_ERR_INVALID_ARG
    assert "n_kv_heads" in D.dflash_last_error()
    a.dims = D.dflash_dims(256, 4, 2, 96, 512, 1000, 1e4, 1e-6, D.DFLASH_BF16)
    assert L.dflash_embed(C.byref(a), None, 0, None) == D.DFLASH_ERR_INVALID_ARG
    assert "head_dim" in D.dflash_last_error()
    # workspace too small
    a.dims = D.dflash_dims(256, 4, 2, 64, 512, 1000, 1e4, 1e-6, D.DFLASH_BF16)
    a.embed, a.first, a.h = 16, 16, 16
    a.n_seqs, a.rows, a.fill_token = 1, 4, 3
    assert L.dflash_embed(C.byref(a), C.c_void_p(256), 16, None) == D.DFLASH_ERR_WORKSPACE
    # verify needs drafts when block > 1
    v = D.dflash_verify_args()
    v.dims = a.dims
    v.h = v.final_norm = v.lm_head = v.argmax = v.accept_len = v.out_tokens = 16
    v.n_seqs, v.block = 1, 4
    assert L.dflash_verify_accept(C.byref(v), C.c_void_p(256), 1 << 30, None) == D.DFLASH_ERR_INVALID_ARG
    assert "drafts" in D.dflash_last_error()
    # workspace sizing is positive for a valid request
    assert D.dflash_workspace_bytes(D.DFLASH_OP_EMBED, a) > 0


def test_binding_raises(D):
    with pytest.raises(D.DFlashError) as e:
        D.dflash_embed(D.dflash_embed_args(), 0, 0, stream=0)
    assert e.value.code == D.DFLASH_ERR_INVALID_ARG


def _qwen_verify(D, S, B):
    v = D.dflash_verify_args()
    v.dims = D.dflash_dims(4096, 32, 8, 128, 12288, 151936, 1e6, 1e-6, D.DFLASH_BF16)
    v.h = v.final_norm = v.lm_head = v.argmax = v.accept_len = v.out_tokens = v.drafts = 256
    v.n_seqs, v.block = S, B
    return v


def test_noalloc_scratch_limit_at_full_shapes(D):
    """Where the allocation-free verification's 8 MiB scratch ends, at the
    Qwen3-8B shapes (H 4096, V 151936): up to 32 token rows per call fit (a
    16- or 17-row block of one sequence, two 16-row blocks), 33 and more do
    not.  Without a GPU the library sizes for its fallback SM count (148),
    a few percent below GB300's 152, where the same rows fit."""
    limit = 8 << 20
    for S, B, fits in ((1, 16, True), (1, 17, True), (2, 16, True), (1, 32, True), (1, 33, False),
                       (4, 16, False), (32, 17, False)):
        need = D.dflash_workspace_bytes(D.DFLASH_OP_VERIFY, _qwen_verify(D, S, B))
        assert need > 0
        assert (need <= limit) == fits, (S, B, need)
        # the documented formula, at 152 SMs (a GB300), keeps the same verdict
        M = S * B
        bn = next(b for b in (16, 32, 64, 128, 256) if b >= min(M, 256))
        G = 152
        formula = 131328 + M * 4096 * 2 + 2 * G * bn * 512 + G * M * 12
        assert (formula + 1024 <= limit) == fits, (S, B, formula)
    # beyond the limit: rejected before any device work, with the size in the message
    rc = D.lib().dflash_verify_accept_noalloc(C.byref(_qwen_verify(D, 4, 16)), None, None)
    assert rc == D.DFLASH_ERR_WORKSPACE
    assert "8 MiB" in D.dflash_last_error()


def test_noalloc_checks_arguments_first(D):
    """Bad arguments give DFLASH_ERR_INVALID_ARG, as dflash_verify_accept
    does, never a scratch-size error; dflash_workspace_bytes gives 0."""
    L = D.lib()
    for field, val, word in (("n_seqs", -3, "n_seqs"), ("block", 0, "block")):
        v = _qwen_verify(D, 1, 16)
        setattr(v, field, val)
        assert L.dflash_verify_accept_noalloc(C.byref(v), None, None) == D.DFLASH_ERR_INVALID_ARG
        assert word in D.dflash_last_error()
        assert D.dflash_workspace_bytes(D.DFLASH_OP_VERIFY, v) == 0
    v = _qwen_verify(D, 1, 16)
    v.dims.dtype = 7
    assert L.dflash_verify_accept_noalloc(C.byref(v), None, None) == D.DFLASH_ERR_INVALID_ARG
    assert "dtype" in D.dflash_last_error()
    v = _qwen_verify(D, 1, 16)
    v.dims.hidden = 4100 - 2  # not a multiple of 8
    assert D.dflash_workspace_bytes(D.DFLASH_OP_VERIFY, v) == 0
    v = _qwen_verify(D, 1, 16)
    v.drafts = 0
    assert L.dflash_verify_accept_noalloc(C.byref(v), None, None) == D.DFLASH_ERR_INVALID_ARG
    assert "drafts" in D.dflash_last_error()


def test_checked_variant_builds_and_exports(D):
    """libdflash_checked.so is built next to the normal library, exports the
    same functions and reports itself as the checked variant."""
    from block_diffusion_speculative_step_gb300 import build
    assert os.path.exists(build.LIB_CHECKED)
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_CHECKED], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    for name in header_functions():
        assert name in exported, name
    chk = C.CDLL(build.LIB_CHECKED)
    chk.dflash_build_flags.restype = C.c_int32
    assert chk.dflash_build_flags() == D.DFLASH_BUILD_CHECKED
    assert D.dflash_build_flags() == 0
