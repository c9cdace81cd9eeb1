"""Displaced-patch-parallel layer step on GB300: thin Python binding of libdpp.so.

The library (``csrc/``, declared in ``include/dpp.h``) does every step of the
path in its own CUDA kernels; this module only marshals torch tensors (device
memory and streams) into the C ABI's plain pointers and sizes, and raises
``DppError`` on a non-zero status.  There is no fallback: if the library has not
been built, every call raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "DppError", "load", "F32", "BF16", "SYNC", "STALE", "LayerParams", "LayerWeights",
    "LayerState", "WorkspaceLayout", "refresh_residual", "halo_conv3x3", "stale_kv_attention",
    "patch_layer_step", "workspace_layout", "workspace_size", "message_sizes",
    "read_device_status", "layer_kernel_count", "status_string", "dtype_code", "alloc_layer",
    "swap_state",
]

F32, BF16 = 0, 1
SYNC, STALE = 0, 1
_c_int, _c_void = ctypes.c_int, ctypes.c_void_p


class DppError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: status {code} ({status_string(code)})")


class LayerParams(ctypes.Structure):
    _fields_ = [("B", _c_int), ("H", _c_int), ("W", _c_int), ("C", _c_int), ("P", _c_int),
                ("G", _c_int), ("heads", _c_int), ("head_dim", _c_int), ("dtype", _c_int),
                ("refresh", _c_int), ("eps", ctypes.c_float), ("gn_mode", _c_int),
                ("fuse_gn", _c_int), ("fuse_refresh", _c_int)]


class LayerWeights(ctypes.Structure):
    _fields_ = [("gamma", _c_void), ("beta", _c_void), ("w_conv", _c_void), ("w_qkv", _c_void),
                ("w_o", _c_void)]


class LayerState(ctypes.Structure):
    _fields_ = [("gn_stats", _c_void), ("y_stale", _c_void), ("k_stale", _c_void),
                ("v_stale", _c_void), ("codes", _c_void), ("scales", _c_void),
                ("gn_next", _c_void), ("y_next", _c_void), ("k_next", _c_void),
                ("v_next", _c_void)]


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("status", "gn_partial", "gn_fresh", "gn_params", "y", "h", "q", "k", "v", "o", "attn_partial",
                 "attn_partial_bytes", "total")]


class OtilParams(ctypes.Structure):
    _fields_ = [(n, _c_int) for n in ("B", "C", "H", "W", "P", "bh", "bw", "k", "dtype")]


_lib = None
EXPORTS = ("dpp_status_string", "dpp_version", "refresh_residual", "halo_conv3x3",
           "stale_kv_attention", "stale_kv_attention_split", "dpp_attention_scratch_size",
           "apply_residual", "dpp_apply_layer_message", "dpp_workspace_query", "dpp_workspace_size", "dpp_message_elems",
           "dpp_message_blocks", "patch_layer_step", "patch_layer_step_timed",
           "dpp_read_device_status", "dpp_layer_kernel_count", "patch_layer_step_noalloc",
           "dpp_noalloc_read_status",
           "dpp_otil_blocks", "dpp_otil_step", "dpp_otil_finalize", "dpp_debug_bounds")


def load(build_if_missing: bool = False):
    """Load libdpp.so (optionally building it first).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise DppError(-1, f"CUDA library not built ({path}); run __graft_entry__.build()")
        _build.build_library()
    _lib = open_library(path)
    return _lib


def open_library(path: str):
    """A ctypes handle on the library at `path` (e.g. the index-checking build), with
    the argument types set; `using(handle)` makes the calls of this module go to it."""
    lib = ctypes.CDLL(path)
    P, I64 = ctypes.POINTER, ctypes.c_int64
    lib.dpp_status_string.restype = ctypes.c_char_p
    lib.dpp_status_string.argtypes = [_c_int]
    lib.dpp_version.restype = _c_int
    lib.refresh_residual.restype = _c_int
    lib.refresh_residual.argtypes = [_c_void, _c_void, _c_void, _c_void, I64, _c_int, _c_void]
    lib.apply_residual.restype = _c_int
    lib.apply_residual.argtypes = [_c_void, _c_void, _c_void, I64, _c_int, _c_void]
    lib.dpp_apply_layer_message.restype = _c_int
    lib.dpp_apply_layer_message.argtypes = [P(LayerParams), _c_void, _c_void, _c_void,
                                            P(LayerState), _c_void]
    lib.halo_conv3x3.restype = _c_int
    lib.halo_conv3x3.argtypes = [_c_void] * 4 + [_c_int] * 7 + [_c_void, _c_void]
    lib.stale_kv_attention.restype = _c_int
    lib.stale_kv_attention.argtypes = ([_c_void] * 6 + [_c_int] * 6 +
                                       [_c_void, ctypes.c_size_t, _c_void, _c_void])
    lib.stale_kv_attention_split.restype = _c_int
    lib.stale_kv_attention_split.argtypes = ([_c_void] * 6 + [_c_int] * 6 +
                                             [_c_void, ctypes.c_size_t, _c_void, _c_void])
    lib.dpp_attention_scratch_size.restype = ctypes.c_size_t
    lib.dpp_attention_scratch_size.argtypes = [_c_int] * 7
    lib.dpp_workspace_query.restype = _c_int
    lib.dpp_workspace_query.argtypes = [P(LayerParams), P(WorkspaceLayout)]
    lib.dpp_workspace_size.restype = ctypes.c_size_t
    lib.dpp_workspace_size.argtypes = [P(LayerParams)]
    lib.dpp_message_elems.restype = I64
    lib.dpp_message_elems.argtypes = [P(LayerParams)]
    lib.dpp_message_blocks.restype = I64
    lib.dpp_message_blocks.argtypes = [P(LayerParams)]
    lib.patch_layer_step.restype = _c_int
    lib.patch_layer_step.argtypes = [P(LayerParams), P(LayerWeights), P(LayerState), _c_void,
                                     _c_void, _c_int, _c_void, _c_void]
    lib.patch_layer_step_timed.restype = _c_int
    lib.patch_layer_step_timed.argtypes = [P(LayerParams), P(LayerWeights), P(LayerState), _c_void,
                                           _c_void, _c_int, _c_void, _c_void, _c_void]
    lib.patch_layer_step_noalloc.restype = _c_int
    lib.patch_layer_step_noalloc.argtypes = [P(LayerParams), P(LayerWeights), P(LayerState),
                                             _c_void, _c_void, _c_int, _c_void]
    lib.dpp_noalloc_read_status.restype = _c_int
    lib.dpp_noalloc_read_status.argtypes = [_c_void]
    lib.dpp_read_device_status.restype = _c_int
    lib.dpp_read_device_status.argtypes = [_c_void, _c_void]
    lib.dpp_otil_blocks.restype = _c_int
    lib.dpp_otil_blocks.argtypes = [P(OtilParams)]
    lib.dpp_otil_step.restype = _c_int
    lib.dpp_otil_step.argtypes = [P(OtilParams)] + [_c_void] * 6
    lib.dpp_otil_finalize.restype = _c_int
    lib.dpp_otil_finalize.argtypes = [P(OtilParams), _c_void, _c_void, _c_void, _c_int, _c_void]
    lib.dpp_layer_kernel_count.restype = _c_int
    lib.dpp_layer_kernel_count.argtypes = [P(LayerParams), _c_int]
    lib.dpp_debug_bounds.restype = _c_int
    lib.dpp_debug_bounds.argtypes = [P(I64), _c_int]
    return lib


@contextlib.contextmanager
def using(lib):
    """Within the block, this module's calls go to the library handle `lib`."""
    global _lib
    prev = load()
    _lib = lib
    try:
        yield lib
    finally:
        _lib = prev


def status_string(code: int) -> str:
    if _lib is None:
        return "library not loaded"
    return _lib.dpp_status_string(code).decode()


def _check(rc: int, where: str):
    if rc != 0:
        raise DppError(rc, where)


def dtype_code(t) -> int:
    dt = t.dtype if isinstance(t, torch.Tensor) else t
    if dt == torch.bfloat16:
        return BF16
    if dt == torch.float32:
        return F32
    raise DppError(4, f"unsupported dtype {dt}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise DppError(1, "tensor is not on a CUDA device")
    if not t.is_contiguous():
        raise DppError(2, "tensor is not contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def refresh_residual(fresh, stale, codes, scales, stream=None):
    """Refresh ``stale`` in place from ``fresh``; writes int8 ``codes`` and fp32 ``scales``."""
    lib = load()
    _check(lib.refresh_residual(_ptr(fresh), _ptr(stale), _ptr(codes), _ptr(scales),
                                fresh.numel(), dtype_code(fresh), _stream(stream)),
           "refresh_residual")


def apply_residual(codes, scales, stale, stream=None):
    """The receiver's half of refresh_residual: stale <- store(fmaf(code, scale, stale))."""
    lib = load()
    _check(lib.apply_residual(_ptr(codes), _ptr(scales), _ptr(stale), stale.numel(),
                              dtype_code(stale), _stream(stream)), "apply_residual")


def apply_layer_message(prm: "LayerParams", codes, scales, gn_sums, copy: dict, stream=None):
    """Applies one stale step's message (codes, scales, the sender's GroupNorm sums) to
    another rank's copy of the layer state (a dict like alloc_layer's)."""
    st = LayerState()
    for k in ("gn_stats", "y_stale", "k_stale", "v_stale"):
        setattr(st, k, _ptr(copy[k]))
    _check(load().dpp_apply_layer_message(ctypes.byref(prm), _ptr(codes), _ptr(scales),
                                          _ptr(gn_sums), ctypes.byref(st), _stream(stream)),
           "dpp_apply_layer_message")


def halo_conv3x3(y_fresh, y_stale, w, out, P: int, dev_status=None, stream=None):
    lib = load()
    B, H, W, Cin = y_fresh.shape
    Cout = w.shape[0]
    _check(lib.halo_conv3x3(_ptr(y_fresh), _ptr(y_stale), _ptr(w), _ptr(out), B, H, W, Cin, Cout,
                            P, dtype_code(y_fresh), _ptr(dev_status), _stream(stream)),
           "halo_conv3x3")


def attention_scratch_size(B: int, L: int, heads: int, P: int, dtype: int = BF16,
                           split: bool = False) -> int:
    """Bytes of the scratch buffer stale_kv_attention (split=False) or
    stale_kv_attention_split (split=True) needs on the current device."""
    return load().dpp_attention_scratch_size(B, L, heads, 64, P, dtype, 1 if split else 0)


def _attention(fn, name, q, k_fresh, v_fresh, k_stale, v_stale, o, heads, P, scratch,
               dev_status, stream, split):
    B, L, C = q.shape
    if scratch is None:
        n = attention_scratch_size(B, L, heads, P, dtype_code(q), split)
        scratch = torch.empty(n, dtype=torch.uint8, device=q.device) if n else None
    nbytes = 0 if scratch is None else scratch.numel() * scratch.element_size()
    _check(fn(_ptr(q), _ptr(k_fresh), _ptr(v_fresh), _ptr(k_stale), _ptr(v_stale), _ptr(o), B, L,
              heads, C // heads, P, dtype_code(q), _ptr(scratch), nbytes, _ptr(dev_status),
              _stream(stream)), name)


def stale_kv_attention(q, k_fresh, v_fresh, k_stale, v_stale, o, heads: int, P: int,
                       scratch=None, dev_status=None, stream=None):
    """Whole units per CTA.  ``scratch``: a device buffer of at least
    attention_scratch_size(split=False) bytes, or None to have one allocated here (by
    torch, the caller's allocator)."""
    _attention(load().stale_kv_attention, "stale_kv_attention", q, k_fresh, v_fresh, k_stale,
               v_stale, o, heads, P, scratch, dev_status, stream, False)


def stale_kv_attention_split(q, k_fresh, v_fresh, k_stale, v_stale, o, heads: int, P: int,
                             scratch=None, dev_status=None, stream=None):
    """stale_kv_attention with the last units shared by all SMs; ``scratch`` as above with
    attention_scratch_size(split=True) bytes."""
    _attention(load().stale_kv_attention_split, "stale_kv_attention_split", q, k_fresh, v_fresh,
               k_stale, v_stale, o, heads, P, scratch, dev_status, stream, True)


GN_SPLICED, GN_SYNC, GN_PREVIOUS = 0, 1, 2


def make_params(B, H, W, C, P, G, heads, dtype, refresh=True, eps=1e-5, head_dim=64,
                gn_mode=GN_SPLICED, fuse_gn=False, fuse_refresh=False):
    return LayerParams(B, H, W, C, P, G, heads, head_dim, dtype, 1 if refresh else 0, eps,
                       gn_mode, 1 if fuse_gn else 0, 1 if fuse_refresh else 0)


def workspace_layout(prm: LayerParams) -> WorkspaceLayout:
    lo = WorkspaceLayout()
    _check(load().dpp_workspace_query(ctypes.byref(prm), ctypes.byref(lo)), "dpp_workspace_query")
    return lo


def workspace_size(prm: LayerParams) -> int:
    return workspace_layout(prm).total


def message_sizes(prm: LayerParams):
    lib = load()
    return lib.dpp_message_elems(ctypes.byref(prm)), lib.dpp_message_blocks(ctypes.byref(prm))


def layer_kernel_count(prm: LayerParams, mode: int) -> int:
    return load().dpp_layer_kernel_count(ctypes.byref(prm), mode)


NUM_STAGE_EVENTS = 7
STAGES = ("groupnorm", "halo_conv", "qkv_proj", "attention", "out_proj", "state_update")
NEXT_KEYS = ("gn_next", "y_next", "k_next", "v_next")
STATE_KEYS = ("gn_stats", "y_stale", "k_stale", "v_stale")


def _layer_state(state: dict) -> "LayerState":
    return LayerState(*[_ptr(state.get(k)) for k in STATE_KEYS + ("codes", "scales") + NEXT_KEYS])


def swap_state(state: dict):
    """After a step that wrote the second state set: makes it the current one."""
    for cur, nxt in zip(STATE_KEYS, NEXT_KEYS):
        state[cur], state[nxt] = state[nxt], state[cur]


def patch_layer_step(prm: LayerParams, weights: dict, state: dict, x, out, mode: int, workspace,
                     stream=None, stage_events=None):
    """One layer pass of all P virtual ranks plus the state update.

    weights: gamma, beta (fp32 [C]), w_conv [C,3,3,C], w_qkv [3C,C], w_o [C,C].
    state:   gn_stats [B,P,G,2] fp32, y_stale [B,H,W,C], k_stale/v_stale [B,L,C],
             codes int8 [message elems], scales fp32 [message blocks]; optionally the
             second set gn_next, y_next, k_next, v_next (see swap_state).
    workspace: uint8 device tensor of workspace_size(prm) bytes.
    """
    lib = load()
    w = LayerWeights(_ptr(weights["gamma"]), _ptr(weights["beta"]), _ptr(weights["w_conv"]),
                     _ptr(weights["w_qkv"]), _ptr(weights["w_o"]))
    s = _layer_state(state)
    if stage_events is None:
        _check(lib.patch_layer_step(ctypes.byref(prm), ctypes.byref(w), ctypes.byref(s), _ptr(x),
                                    _ptr(out), mode, _ptr(workspace), _stream(stream)),
               "patch_layer_step")
        return
    if len(stage_events) != NUM_STAGE_EVENTS:
        raise DppError(9, "stage_events needs 7 torch.cuda.Event objects")
    evs = (ctypes.c_void_p * NUM_STAGE_EVENTS)(*[e.cuda_event for e in stage_events])
    _check(lib.patch_layer_step_timed(ctypes.byref(prm), ctypes.byref(w), ctypes.byref(s),
                                      _ptr(x), _ptr(out), mode, _ptr(workspace), _stream(stream),
                                      evs),
           "patch_layer_step_timed")


def patch_layer_step_noalloc(prm: LayerParams, weights: dict, state: dict, x, out, mode: int,
                             stream=None):
    """patch_layer_step with the library's fixed 80 MiB device scratch as workspace.

    For callers that cannot allocate device memory when they run a layer; nothing
    is allocated here or in the library.  Calls that overlap on the GPU share the
    scratch and race; the first call on a device should precede any stream capture.
    """
    lib = load()
    w = LayerWeights(_ptr(weights["gamma"]), _ptr(weights["beta"]), _ptr(weights["w_conv"]),
                     _ptr(weights["w_qkv"]), _ptr(weights["w_o"]))
    s = _layer_state(state)
    _check(lib.patch_layer_step_noalloc(ctypes.byref(prm), ctypes.byref(w), ctypes.byref(s),
                                        _ptr(x), _ptr(out), mode, _stream(stream)),
           "patch_layer_step_noalloc")


def read_device_status(workspace, stream=None) -> int:
    return load().dpp_read_device_status(_ptr(workspace), _stream(stream))


def debug_bounds(reset: bool = False):
    """(code, record) of the index-checking build's first out-of-extent index (see
    dpp_debug_bounds): code DPP_OK / DPP_ERR_BOUNDS (7) / DPP_ERR_UNSUPPORTED (8, a normal
    build); record = (file, line, index, extent)."""
    rec = (ctypes.c_int64 * 4)()
    rc = load().dpp_debug_bounds(rec, 1 if reset else 0)
    return rc, tuple(rec)


def noalloc_read_status(stream=None) -> int:
    """Device status word of the last patch_layer_step_noalloc on the current device."""
    return load().dpp_noalloc_read_status(_stream(stream))


# ------------------------------------------------------------------ helpers for callers
def alloc_layer(prm: LayerParams, device="cuda", double_buffer=False):
    """Allocates (with torch) the state, message and workspace of one layer; with
    double_buffer also the second state set the step writes (gn_next, y_next, k_next,
    v_next), to be swapped in after each step that writes it (swap_state)."""
    dt = torch.bfloat16 if prm.dtype == BF16 else torch.float32
    B, H, W, C, P, G = prm.B, prm.H, prm.W, prm.C, prm.P, prm.G
    n_codes, n_scales = message_sizes(prm)
    state = dict(
        gn_stats=torch.zeros(B, P, G, 2, dtype=torch.float32, device=device),
        y_stale=torch.zeros(B, H, W, C, dtype=dt, device=device),
        k_stale=torch.zeros(B, H * W, C, dtype=dt, device=device),
        v_stale=torch.zeros(B, H * W, C, dtype=dt, device=device),
        codes=torch.zeros(n_codes, dtype=torch.int8, device=device),
        scales=torch.zeros(n_scales, dtype=torch.float32, device=device),
    )
    if double_buffer:
        for cur, nxt in zip(STATE_KEYS, NEXT_KEYS):
            state[nxt] = torch.zeros_like(state[cur])
    ws = torch.zeros(workspace_size(prm), dtype=torch.uint8, device=device)
    return state, ws


def workspace_views(prm: LayerParams, ws):
    """Typed views of the workspace pieces (for inspection and tests)."""
    lo = workspace_layout(prm)
    dt = torch.bfloat16 if prm.dtype == BF16 else torch.float32
    es = 2 if prm.dtype == BF16 else 4
    B, H, W, C, P, G = prm.B, prm.H, prm.W, prm.C, prm.P, prm.G
    n = B * H * W * C

    def view(off, count, dtype, shape):
        return ws[off:off + count * (torch.finfo(dtype).bits // 8)].view(dtype).view(*shape)

    out = dict(gn_fresh=view(lo.gn_fresh, B * P * G * 2, torch.float32, (B, P, G, 2)),
               y=view(lo.y, n, dt, (B, H, W, C)), h=view(lo.h, n, dt, (B, H, W, C)))
    if prm.fuse_gn:
        out["gn_params"] = view(lo.gn_params, B * P * 3 * C, torch.float32, (B, P, 3, C))
    for name in ("q", "k", "v", "o"):
        out[name] = view(getattr(lo, name), n, dt, (B, H * W, C))
    assert es in (2, 4)
    return out


# ------------------------------------------------------------------ OTIL exchange
def otil_params(B, C, H, W, P, bh, bw, k, dtype=BF16) -> OtilParams:
    return OtilParams(B, C, H, W, P, bh, bw, k, dtype)


def otil_blocks(prm: OtilParams) -> int:
    """Sub-blocks per band (K), or -1 for invalid params."""
    return load().dpp_otil_blocks(ctypes.byref(prm))


def otil_alloc(prm: OtilParams, fresh0, device="cuda"):
    """The exchange state: every rank's view initialised to fresh0 [B,C,H,W], cleared
    flags, and the selection / message outputs."""
    K = otil_blocks(prm)
    if K < 0:
        raise DppError(2, "invalid OTIL params")
    dt = fresh0.dtype
    views = fresh0.to(device).unsqueeze(0).repeat(prm.P, 1, 1, 1, 1).contiguous()
    visited = torch.zeros(prm.P, K, dtype=torch.uint8, device=device)
    sel = torch.zeros(prm.P, prm.k, dtype=torch.int32, device=device)
    msg = torch.zeros(prm.P, prm.k, prm.B, prm.C, prm.bh, prm.bw, dtype=dt, device=device)
    return dict(views=views, visited=visited, sel=sel, msg=msg)


def otil_step(prm: OtilParams, fresh, st: dict, stream=None):
    _check(load().dpp_otil_step(ctypes.byref(prm), _ptr(fresh), _ptr(st["views"]),
                                _ptr(st["visited"]), _ptr(st["sel"]), _ptr(st["msg"]),
                                _stream(stream)), "dpp_otil_step")


def otil_finalize(prm: OtilParams, fresh, st: dict, reset: bool = False, stream=None):
    _check(load().dpp_otil_finalize(ctypes.byref(prm), _ptr(fresh), _ptr(st["views"]),
                                    _ptr(st["visited"]), 1 if reset else 0, _stream(stream)),
           "dpp_otil_finalize")
