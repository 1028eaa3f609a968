"""ctypes binding of the C ABI in include/dflash.h: the same struct and
function names, argument marshalling only.  Raises DFlashError on a
non-zero status.  There is no fallback: if libdflash.so is missing the
import fails loudly."""
from __future__ import annotations

import ctypes as C
import os

from . import build as _build

DFLASH_OK = 0
DFLASH_ERR_INVALID_ARG = -1
DFLASH_ERR_UNSUPPORTED = -2
DFLASH_ERR_WORKSPACE = -3
DFLASH_ERR_CUDA = -4
DFLASH_ERR_TIMEOUT = -5
DFLASH_ERR_NUMERIC = -6
DFLASH_ERR_CHECK = -7

DFLASH_F32 = 0
DFLASH_BF16 = 1
DFLASH_ATTN_CAUSAL = 0
DFLASH_ATTN_BLOCK_BIDIR = 1
(DFLASH_OP_EMBED, DFLASH_OP_LAYER, DFLASH_OP_FUSE, DFLASH_OP_DRAFT, DFLASH_OP_VERIFY, DFLASH_OP_PATH,
 DFLASH_OP_SAMPLE_DRAFTS, DFLASH_OP_SAMPLE_ACCEPT) = range(8)
DFLASH_MAX_LAYERS = 16

# Every symbol the header exports (checked by the CPU test suite).
EXPORTS = ("dflash_rope_table", "dflash_embed", "dflash_decoder_layer_forward", "dflash_fuse_context",
           "dflash_draft_block", "dflash_verify_accept", "dflash_path_select", "dflash_workspace_bytes",
           "dflash_workspace_init", "dflash_read_status", "dflash_last_error", "dflash_abi_version",
           "dflash_trace_begin", "dflash_trace_pause", "dflash_trace_read", "dflash_trace_end",
           "dflash_verify_accept_noalloc", "dflash_trace_launches", "dflash_sample_drafts",
           "dflash_sample_accept", "dflash_workspace_control", "dflash_build_flags")
DFLASH_TRACE_FAMILIES = 13


class DFlashError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"dflash error {code}: {msg}")
        self.code = code


vp = C.c_void_p
i32 = C.c_int32
f32 = C.c_float
P_i32 = C.POINTER(C.c_int32)
P_f32 = C.POINTER(C.c_float)


class dflash_dims(C.Structure):
    _fields_ = [("hidden", i32), ("n_q_heads", i32), ("n_kv_heads", i32), ("head_dim", i32),
                ("intermediate", i32), ("vocab", i32), ("rope_theta", f32), ("rms_eps", f32), ("dtype", i32)]


class dflash_kv(C.Structure):
    _fields_ = [("k", vp), ("v", vp), ("capacity", i32), ("window", i32), ("pages", vp), ("page_size", i32),
                ("max_pages", i32), ("pool_pages", i32)]


class dflash_layer_weights(C.Structure):
    _fields_ = [("w_qkv", vp), ("w_o", vp), ("w_gu", vp), ("w_down", vp), ("ln1", vp), ("ln2", vp)]


class dflash_embed_args(C.Structure):
    _fields_ = [("dims", dflash_dims), ("embed", vp), ("n_seqs", i32), ("rows", i32), ("first", vp),
                ("rest", vp), ("fill_token", i32), ("h", vp)]


class dflash_layer_args(C.Structure):
    _fields_ = [("dims", dflash_dims), ("w", dflash_layer_weights), ("n_seqs", i32), ("rows", i32),
                ("base_pos", vp), ("h", vp), ("kv", dflash_kv), ("attn_mode", i32), ("max_pos", i32),
                ("rope_cs", vp), ("rope_max_pos", i32), ("tap", vp), ("tap_stride", i32),
                ("tap_offset", i32), ("out_x_attn", vp), ("out_q", vp), ("out_kb", vp), ("out_vb", vp),
                ("out_attn", vp), ("out_x_mlp", vp), ("out_act", vp)]


class dflash_fuse_args(C.Structure):
    _fields_ = [("dims", dflash_dims), ("n_taps", i32), ("w_fc", vp), ("fc_norm", vp), ("n_layers", i32),
                ("w_qkv_layers", vp * DFLASH_MAX_LAYERS), ("kv_layers", dflash_kv * DFLASH_MAX_LAYERS),
                ("feats", vp), ("n_seqs", i32), ("rows", i32), ("base_pos", vp), ("valid", vp),
                ("rope_cs", vp), ("rope_max_pos", i32), ("c_out", vp)]


class dflash_draft_args(C.Structure):
    _fields_ = [("dims", dflash_dims), ("n_layers", i32), ("layers", dflash_layer_weights * DFLASH_MAX_LAYERS),
                ("kv_layers", dflash_kv * DFLASH_MAX_LAYERS), ("final_norm", vp), ("embed", vp),
                ("lm_head", vp), ("n_seqs", i32), ("block", i32), ("anchor", vp), ("base_pos", vp),
                ("mask_token", i32), ("max_pos", i32), ("rope_cs", vp), ("rope_max_pos", i32),
                ("drafts", vp), ("logits", vp), ("path_topk", i32), ("path_rank", i32), ("path_u", vp),
                ("path_v", vp), ("denoise_rounds", i32), ("path_temperature", C.c_float), ("path_seed", C.c_uint64),
                ("path_cycle", i32), ("path_cand_out", vp), ("path_logq", vp), ("conv_rank", i32),
                ("conv_w1", vp * DFLASH_MAX_LAYERS), ("conv_w2", vp * DFLASH_MAX_LAYERS)]


class dflash_verify_args(C.Structure):
    _fields_ = [("dims", dflash_dims), ("h", vp), ("final_norm", vp), ("lm_head", vp), ("n_seqs", i32),
                ("block", i32), ("drafts", vp), ("argmax", vp), ("margin", vp), ("accept_len", vp),
                ("out_tokens", vp), ("next_anchor", vp), ("base_pos", vp), ("commit_base", vp),
                ("commit_count", vp), ("logits", vp)]


class dflash_path_args(C.Structure):
    _fields_ = [("dims", dflash_dims), ("n_seqs", i32), ("block", i32), ("topk", i32), ("rank", i32),
                ("embed", vp), ("path_u", vp), ("path_v", vp), ("anchor", vp), ("cand", vp), ("path", vp),
                ("margin", vp), ("temperature", C.c_float), ("seed", C.c_uint64), ("cycle", i32), ("base_pos", vp),
                ("logq", vp)]


class dflash_sample_drafts_args(C.Structure):
    _fields_ = [("dims", dflash_dims), ("n_seqs", i32), ("block", i32), ("temperature", C.c_float),
                ("cycle", i32), ("seed", C.c_uint64), ("base_pos", vp), ("draft_logits", vp), ("drafts", vp),
                ("draft_lse", vp), ("top_k", i32), ("top_p", C.c_float)]


class dflash_sample_accept_args(C.Structure):
    _fields_ = [("dims", dflash_dims), ("n_seqs", i32), ("block", i32), ("temperature", C.c_float),
                ("cycle", i32), ("seed", C.c_uint64), ("target_logits", vp), ("draft_logits", vp),
                ("draft_lse", vp), ("drafts", vp), ("base_pos", vp), ("update_base_pos", i32),
                ("accept_len", vp), ("out_tokens", vp), ("next_anchor", vp), ("commit_base", vp),
                ("commit_count", vp), ("top_k", i32), ("top_p", C.c_float), ("draft_topk", i32),
                ("draft_cand", vp), ("draft_logq", vp)]


class dflash_trace_stat(C.Structure):
    _fields_ = [("name", C.c_char * 24), ("launches", i32), ("total_ms", C.c_double), ("bytes", C.c_double)]


_lib = None


def lib(path: str | None = None):
    """Load libdflash.so (built in-tree by __graft_entry__.build()), or the
    checked variant libdflash_checked.so when DFLASH_LIB=checked is set."""
    global _lib
    if _lib is None:
        path = path or (_build.LIB_CHECKED if os.environ.get("DFLASH_LIB") == "checked" else _build.LIB)
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first (__graft_entry__.build())")
        L = C.CDLL(path)
        for name in ("dflash_embed", "dflash_decoder_layer_forward", "dflash_fuse_context", "dflash_draft_block",
                     "dflash_verify_accept", "dflash_path_select", "dflash_sample_drafts", "dflash_sample_accept"):
            getattr(L, name).argtypes = [vp, vp, C.c_size_t, vp]
            getattr(L, name).restype = C.c_int
        L.dflash_rope_table.argtypes = [f32, i32, i32, vp, vp]
        L.dflash_rope_table.restype = C.c_int
        L.dflash_workspace_bytes.argtypes = [i32, vp]
        L.dflash_workspace_bytes.restype = C.c_size_t
        L.dflash_workspace_init.argtypes = [vp, C.c_size_t, vp]
        L.dflash_workspace_init.restype = C.c_int
        L.dflash_workspace_control.argtypes = [vp, C.c_size_t, C.c_uint64, i32, vp]
        L.dflash_workspace_control.restype = C.c_int
        L.dflash_read_status.argtypes = [vp, vp, P_i32]
        L.dflash_read_status.restype = C.c_int
        L.dflash_last_error.restype = C.c_char_p
        L.dflash_abi_version.restype = i32
        L.dflash_build_flags.restype = i32
        L.dflash_trace_begin.argtypes = [i32]
        L.dflash_verify_accept_noalloc.argtypes = [vp, vp, vp]
        L.dflash_verify_accept_noalloc.restype = C.c_int
        L.dflash_trace_read.argtypes = [C.POINTER(dflash_trace_stat), i32]
        L.dflash_trace_launches.argtypes = [vp, vp, i32]
        _lib = L
    return _lib


def _check(rc: int):
    if rc != DFLASH_OK:
        raise DFlashError(rc, lib().dflash_last_error().decode())


def _stream(stream) -> int:
    """Raw cudaStream_t of a torch stream (or an int handle)."""
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


DFLASH_BUILD_CHECKED = 1


def dflash_build_flags() -> int:
    return int(lib().dflash_build_flags())


def dflash_abi_version() -> int:
    return int(lib().dflash_abi_version())


def dflash_last_error() -> str:
    return lib().dflash_last_error().decode()


def dflash_rope_table(theta: float, head_dim: int, max_pos: int, cos_sin_ptr: int, stream=None):
    _check(lib().dflash_rope_table(theta, head_dim, max_pos, cos_sin_ptr, _stream(stream)))


def dflash_workspace_bytes(op: int, args) -> int:
    return int(lib().dflash_workspace_bytes(op, C.byref(args)))


def dflash_workspace_init(ws_ptr: int, ws_bytes: int, stream=None):
    _check(lib().dflash_workspace_init(ws_ptr, ws_bytes, _stream(stream)))


def dflash_workspace_control(ws_ptr: int, ws_bytes: int, wait_limit_ns: int = 0, stall_kv_loads: bool = False,
                             stream=None):
    # stall_kv_loads: True / 1 stalls the attention's K/V copies, 2 the paired GEMM's weight copies
    _check(lib().dflash_workspace_control(ws_ptr, ws_bytes, wait_limit_ns, int(stall_kv_loads),
                                          _stream(stream)))


def dflash_read_status(ws_ptr: int, stream=None) -> int:
    st = C.c_int32(0)
    _check(lib().dflash_read_status(ws_ptr, _stream(stream), C.byref(st)))
    return int(st.value)


def _call(name: str, args, ws_ptr: int, ws_bytes: int, stream):
    _check(getattr(lib(), name)(C.byref(args), ws_ptr, ws_bytes, _stream(stream)))


def dflash_embed(args: dflash_embed_args, ws_ptr: int, ws_bytes: int, stream=None):
    _call("dflash_embed", args, ws_ptr, ws_bytes, stream)


def dflash_decoder_layer_forward(args: dflash_layer_args, ws_ptr: int, ws_bytes: int, stream=None):
    _call("dflash_decoder_layer_forward", args, ws_ptr, ws_bytes, stream)


def dflash_fuse_context(args: dflash_fuse_args, ws_ptr: int, ws_bytes: int, stream=None):
    _call("dflash_fuse_context", args, ws_ptr, ws_bytes, stream)


def dflash_draft_block(args: dflash_draft_args, ws_ptr: int, ws_bytes: int, stream=None):
    _call("dflash_draft_block", args, ws_ptr, ws_bytes, stream)


def dflash_verify_accept(args: dflash_verify_args, ws_ptr: int, ws_bytes: int, stream=None):
    _call("dflash_verify_accept", args, ws_ptr, ws_bytes, stream)


def dflash_verify_accept_noalloc(args: dflash_verify_args, status_ptr: int = 0, stream=None):
    """dflash_verify_accept with the library's fixed 8 MiB device scratch
    instead of a workspace (for callers that cannot allocate)."""
    _check(lib().dflash_verify_accept_noalloc(C.byref(args), status_ptr, _stream(stream)))


def dflash_path_select(args: dflash_path_args, ws_ptr: int, ws_bytes: int, stream=None):
    _call("dflash_path_select", args, ws_ptr, ws_bytes, stream)


def dflash_sample_drafts(args: dflash_sample_drafts_args, ws_ptr: int, ws_bytes: int, stream=None):
    _call("dflash_sample_drafts", args, ws_ptr, ws_bytes, stream)


def dflash_sample_accept(args: dflash_sample_accept_args, ws_ptr: int, ws_bytes: int, stream=None):
    _call("dflash_sample_accept", args, ws_ptr, ws_bytes, stream)


def dflash_trace_begin(max_launches: int = 4096):
    _check(lib().dflash_trace_begin(max_launches))


def dflash_trace_pause():
    _check(lib().dflash_trace_pause())


def dflash_trace_read() -> dict:
    """Per kernel family: {name: (launches, total_ms, bytes)} of the last traced work."""
    arr = (dflash_trace_stat * DFLASH_TRACE_FAMILIES)()
    n = lib().dflash_trace_read(arr, DFLASH_TRACE_FAMILIES)
    if n < 0:
        _check(n)
    return {a.name.decode(): (int(a.launches), float(a.total_ms), float(a.bytes)) for a in arr[:n]}


def dflash_trace_launches() -> list:
    """[(family index, ms)] for every traced launch, in launch order."""
    n = lib().dflash_trace_launches(None, None, 0)
    if n < 0:
        _check(n)
    ms = (C.c_float * max(n, 1))()
    fam = (C.c_int32 * max(n, 1))()
    _check(0 if lib().dflash_trace_launches(ms, fam, n) >= 0 else DFLASH_ERR_CUDA)
    return [(int(fam[i]), float(ms[i])) for i in range(n)]


def dflash_trace_end():
    _check(lib().dflash_trace_end())
