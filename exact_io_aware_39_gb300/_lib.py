"""ctypes binding of libflashattn.so: the C ABI of include/flash_attn.h under
the same names, plus thin helpers that take torch tensors.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI. There is no CPU or PyTorch fallback; if the shared
library is missing or does not load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libflashattn.so")

FA_OK = 0
STATUS_NAMES = {
    0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_WORKSPACE",
    4: "FA_ERR_CUDA", 5: "FA_ERR_DEVICE_TIMEOUT", 6: "FA_ERR_DEVICE_INTERNAL",
    7: "FA_ERR_SCRATCH_LIMIT",
}
FA_ERR_SCRATCH_LIMIT = 7
BWD_NOALLOC_SCRATCH_BYTES = 64 << 20

# every symbol include/flash_attn.h and include/standard_attn.h declare
EXPORTS = [
    "flash_attn_fwd", "flash_attn_fwd_ex", "flash_attn_bwd_workspace_size", "flash_attn_bwd",
    "flash_attn_bwd_ex", "flash_attn_bwd_noalloc",
    "flash_attn_tile_map",
    "flash_attn_get_device_error", "flash_attn_set_profile_events", "flash_attn_status_string",
    "flash_attn_version",
    "standard_attn_workspace_size", "standard_attn_fwd", "standard_attn_bwd",
]


FA_DTYPE_BF16, FA_DTYPE_F16 = 0, 1


class fa_options(ctypes.Structure):
    """Mirror of the C struct fa_options (size is set by the constructor)."""
    _fields_ = [("size", ctypes.c_uint32), ("dtype", ctypes.c_int32), ("p_drop", ctypes.c_float),
                ("reserved", ctypes.c_uint32), ("seed", ctypes.c_uint64),
                ("tile_record", ctypes.c_void_p), ("wait_limit_us", ctypes.c_uint32),
                ("test_stall", ctypes.c_uint32)]

    def __init__(self, dtype=FA_DTYPE_BF16, p_drop=0.0, seed=0, tile_record=None, wait_limit_us=0,
                 test_stall=0):
        super().__init__(ctypes.sizeof(fa_options), dtype, float(p_drop), 0, int(seed), tile_record,
                         int(wait_limit_us), int(test_stall))


class FlashAttnError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


_lib = None


def load(path=LIB_PATH):
    """Loads (once) and returns the ctypes handle of the library."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m exact_io_aware_39_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.flash_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, vp, vp, vp]
    lib.flash_attn_fwd.restype = i32
    opt_p = ctypes.POINTER(fa_options)
    lib.flash_attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, vp, vp, opt_p, vp]
    lib.flash_attn_fwd_ex.restype = i32
    lib.flash_attn_bwd_ex.argtypes = [vp] * 9 + [i32, i32, i32, i32, f32, i32, vp, vp, opt_p, vp, sz, vp]
    lib.flash_attn_bwd_ex.restype = i32
    lib.flash_attn_bwd_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.flash_attn_bwd_workspace_size.restype = sz
    lib.flash_attn_bwd.argtypes = [vp] * 9 + [i32, i32, i32, i32, f32, i32, vp, vp, vp, sz, vp]
    lib.flash_attn_bwd.restype = i32
    lib.flash_attn_bwd_noalloc.argtypes = [vp] * 9 + [i32, i32, i32, i32, f32, i32, vp, vp, vp]
    lib.flash_attn_bwd_noalloc.restype = i32
    lib.flash_attn_tile_map.argtypes = [i32, i32, i32, vp, vp, vp, vp]
    lib.flash_attn_tile_map.restype = i32
    lib.flash_attn_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.flash_attn_get_device_error.restype = i32
    lib.flash_attn_set_profile_events.argtypes = [vp, vp]
    lib.flash_attn_set_profile_events.restype = i32
    lib.flash_attn_status_string.argtypes = [i32]
    lib.flash_attn_status_string.restype = ctypes.c_char_p
    lib.flash_attn_version.argtypes = []
    lib.flash_attn_version.restype = i32
    lib.standard_attn_workspace_size.argtypes = [i32, i32, i32]
    lib.standard_attn_workspace_size.restype = sz
    lib.standard_attn_fwd.argtypes = [vp] * 5 + [i32, i32, i32, i32, f32, i32, vp, vp, opt_p, i32, vp, sz, vp]
    lib.standard_attn_fwd.restype = i32
    lib.standard_attn_bwd.argtypes = [vp] * 7 + [i32, i32, i32, i32, f32, opt_p, i32, vp, sz, vp]
    lib.standard_attn_bwd.restype = i32
    _lib = lib
    return lib


# ---------------------------------------------------------------------------
# raw C-ABI calls (same names and argument order as the header)
# ---------------------------------------------------------------------------

def flash_attn_fwd(Q, K, V, O, LSE, B, H, N, d, scale, causal, kv_len, block_mask, stream):
    return load().flash_attn_fwd(Q, K, V, O, LSE, B, H, N, d, scale, causal, kv_len, block_mask, stream)


def flash_attn_fwd_ex(Q, K, V, O, LSE, B, H, N, d, scale, causal, kv_len, block_mask, options, stream):
    return load().flash_attn_fwd_ex(Q, K, V, O, LSE, B, H, N, d, scale, causal, kv_len, block_mask,
                                    None if options is None else ctypes.byref(options), stream)


def flash_attn_bwd_ex(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal, kv_len, block_mask,
                      options, workspace, workspace_bytes, stream):
    return load().flash_attn_bwd_ex(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal, kv_len,
                                    block_mask, None if options is None else ctypes.byref(options),
                                    workspace, workspace_bytes, stream)


def flash_attn_bwd_workspace_size(B, H, N, d):
    return load().flash_attn_bwd_workspace_size(B, H, N, d)


def flash_attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal, kv_len, block_mask,
                   workspace, workspace_bytes, stream):
    return load().flash_attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal, kv_len,
                                 block_mask, workspace, workspace_bytes, stream)


def flash_attn_bwd_noalloc(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal, kv_len,
                           block_mask, stream):
    """Backward without a workspace argument: for callers that cannot allocate
    device memory (see the header); scratch comes from a fixed 64 MiB array."""
    return load().flash_attn_bwd_noalloc(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal,
                                         kv_len, block_mask, stream)


def flash_attn_tile_map(B, N, causal, kv_len, block_mask, out, stream):
    return load().flash_attn_tile_map(B, N, causal, kv_len, block_mask, out, stream)


def flash_attn_get_device_error():
    detail = (ctypes.c_uint32 * 4)()
    st = load().flash_attn_get_device_error(detail)
    return st, list(detail)


def flash_attn_set_profile_events(start_event, stop_event):
    return load().flash_attn_set_profile_events(start_event, stop_event)


def flash_attn_status_string(status):
    return load().flash_attn_status_string(status).decode()


def flash_attn_version():
    return load().flash_attn_version()


def standard_attn_workspace_size(B, H, N):
    return load().standard_attn_workspace_size(B, H, N)


STANDARD_ATTN_S16 = 1


def standard_attn_fwd(Q, K, V, O, LSE, B, H, N, d, scale, causal, kv_len, block_mask, options, flags, workspace,
                      workspace_bytes, stream):
    return load().standard_attn_fwd(Q, K, V, O, LSE, B, H, N, d, scale, causal, kv_len, block_mask,
                                    None if options is None else ctypes.byref(options), flags, workspace,
                                    workspace_bytes, stream)


def standard_attn_bwd(Q, K, V, dO, dQ, dK, dV, B, H, N, d, scale, options, flags, workspace, workspace_bytes,
                      stream):
    return load().standard_attn_bwd(Q, K, V, dO, dQ, dK, dV, B, H, N, d, scale,
                                    None if options is None else ctypes.byref(options), flags, workspace,
                                    workspace_bytes, stream)


# ---------------------------------------------------------------------------
# torch helpers (device memory and streams come from PyTorch)
# ---------------------------------------------------------------------------

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(st, where):
    if st != FA_OK:
        raise FlashAttnError(st, where)


def _check_inputs(*ts):
    """Validates the tensors and returns the fa_options for their dtype."""
    import torch
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
    dt = ts[0].dtype
    if dt not in (torch.bfloat16, torch.float16):
        raise ValueError("Q, K, V must be bfloat16 or float16 [B, H, N, d]")
    for t in ts:
        if t is not None and (t.dtype != dt or t.dim() != 4):
            raise ValueError("Q, K, V (and O, dO) must share one 16-bit dtype and be [B, H, N, d]")
    return fa_options(FA_DTYPE_F16 if dt == torch.float16 else FA_DTYPE_BF16)


def _mask_args(kv_len, block_mask):
    import torch
    if kv_len is not None and (kv_len.dtype != torch.int32 or not kv_len.is_cuda):
        raise ValueError("kv_len must be a CUDA int32 tensor [B]")
    if block_mask is not None and (block_mask.dtype != torch.uint8 or not block_mask.is_cuda):
        raise ValueError("block_mask must be a CUDA uint8 tensor [nT, nT]")
    return _ptr(kv_len), _ptr(block_mask)


def _set_checks(opts, tile_record, wait_limit_us, test_stall):
    """Fills the checking fields of fa_options: tile_record (a zeroed CUDA
    uint8 tensor [B, H, nT, nT] or None), wait_limit_us, test_stall."""
    import torch
    if tile_record is not None:
        if tile_record.dtype != torch.uint8 or not tile_record.is_cuda or not tile_record.is_contiguous():
            raise ValueError("tile_record must be a contiguous CUDA uint8 tensor [B, H, nT, nT]")
        opts.tile_record = tile_record.data_ptr()
    opts.wait_limit_us = int(wait_limit_us)
    opts.test_stall = int(test_stall)


def attention_fwd(q, k, v, scale, causal=False, kv_len=None, block_mask=None, out=None, lse=None,
                  stream=None, p_drop=0.0, seed=0, tile_record=None, wait_limit_us=0, test_stall=0):
    """O, LSE = attention(q, k, v) on the GPU. q, k, v: bf16 or fp16 [B, H, N, d];
    p_drop > 0 applies dropout to P (mask from Philox4x32-10 keyed by seed).
    tile_record, wait_limit_us and test_stall are the checking options of
    fa_options (see include/flash_attn.h)."""
    import torch
    opts = _check_inputs(q, k, v)
    opts.p_drop, opts.seed = float(p_drop), int(seed)
    _set_checks(opts, tile_record, wait_limit_us, test_stall)
    B, H, N, d = q.shape
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    kv_p, bm_p = _mask_args(kv_len, block_mask)
    st = flash_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, H, N, d, float(scale),
                           int(bool(causal)), kv_p, bm_p, opts, _stream(stream))
    _check(st, "flash_attn_fwd_ex")
    return o, l


def attention_bwd(q, k, v, o, do, lse, scale, causal=False, kv_len=None, block_mask=None,
                  workspace=None, dq=None, dk=None, dv=None, stream=None, p_drop=0.0, seed=0,
                  tile_record=None, wait_limit_us=0, test_stall=0):
    """dQ, dK, dV of attention on the GPU (recomputing S, P and the dropout
    mask on chip); p_drop and seed must match the forward call."""
    import torch
    opts = _check_inputs(q, k, v, o, do)
    opts.p_drop, opts.seed = float(p_drop), int(seed)
    _set_checks(opts, tile_record, wait_limit_us, test_stall)
    B, H, N, d = q.shape
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = flash_attn_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    kv_p, bm_p = _mask_args(kv_len, block_mask)
    st = flash_attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                           _ptr(dv), B, H, N, d, float(scale), int(bool(causal)), kv_p, bm_p, opts,
                           _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "flash_attn_bwd_ex")
    return dq, dk, dv


def tile_map(B, N, causal=False, kv_len=None, block_mask=None, device="cuda", stream=None):
    """uint8 [B, nT, nT] tile states the kernels use (0 skip, 1 full, 2 partial)."""
    import torch
    nT = (N + 127) // 128
    out = torch.empty((B, nT, nT), dtype=torch.uint8, device=device)
    kv_p, bm_p = _mask_args(kv_len, block_mask)
    st = flash_attn_tile_map(B, N, int(bool(causal)), kv_p, bm_p, _ptr(out), _stream(stream))
    _check(st, "flash_attn_tile_map")
    return out


def profile_next_call(start, stop):
    """Record torch.cuda.Event start/stop around the dominant kernel of the
    next attention_fwd/attention_bwd call of this thread."""
    st = flash_attn_set_profile_events(ctypes.c_void_p(start.cuda_event), ctypes.c_void_p(stop.cuda_event))
    _check(st, "flash_attn_set_profile_events")


def device_error():
    """(status, [code, site, block, thread]) of the device error word; clears it."""
    return flash_attn_get_device_error()


def standard_attention_fwd(q, k, v, scale, causal=False, kv_len=None, block_mask=None, workspace=None,
                           stream=None, s16=False):
    """Standard (materialising) attention on the GPU: (O, LSE, workspace); the
    workspace holds S and P and must be passed to standard_attention_bwd.
    s16=True stores S (and later dP) in the 16-bit input type."""
    import torch
    opts = _check_inputs(q, k, v)
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    need = standard_attn_workspace_size(B, H, N)
    if need == 0:
        raise FlashAttnError(2, "standard_attn_workspace_size")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    kv_p, bm_p = _mask_args(kv_len, block_mask)
    st = standard_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, H, N, d, float(scale),
                           int(bool(causal)), kv_p, bm_p, opts, STANDARD_ATTN_S16 if s16 else 0, _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "standard_attn_fwd")
    return o, l, workspace


def standard_attention_bwd(q, k, v, do, workspace, scale, stream=None, s16=False):
    """dQ, dK, dV of standard attention from the P the forward call stored
    (s16 as in the forward call)."""
    import torch
    opts = _check_inputs(q, k, v, do)
    B, H, N, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = standard_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d,
                           float(scale), opts, STANDARD_ATTN_S16 if s16 else 0, _ptr(workspace),
                           workspace.numel() * workspace.element_size(),
                           _stream(stream))
    _check(st, "standard_attn_bwd")
    return dq, dk, dv
