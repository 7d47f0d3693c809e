"""Python binding of the C-ABI attention library (argument marshalling only).

The functions with the C names (``attn_fwd``, ``attn_fwd_varlen``,
``attn_fwd_paged``, ``attn_fwd_fp8``, ``attn_fwd_splitkv``,
``attn_fwd_splitkv_noalloc``, ``attn_lse_merge``, ``attn_bwd``, the status and
self-test calls) take raw device addresses and sizes exactly like
``include/attn.h``.  ``forward``, ``forward_varlen``, ``forward_paged``,
``forward_fp8``, ``forward_splitkv``, ``lse_merge`` and ``backward`` are the
torch-facing conveniences: they check dtypes / devices / contiguity, allocate
the outputs (and any workspace) with torch, and call the library on the
current CUDA stream.  Every step of the computation runs in
the library's CUDA kernel; there is no CPU fallback, and a missing library is
an error.
"""

from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libattn.so")
_lib = None

ATTN_OK = 0
ATTN_ERR_NULLPTR = 1
ATTN_ERR_ALIGN = 2
ATTN_ERR_SHAPE = 3
ATTN_ERR_UNSUPPORTED_D = 4
ATTN_ERR_SCALE = 5
ATTN_ERR_CUDA = 6
ATTN_ERR_DEVICE_TIMEOUT = 7
ATTN_ERR_UNSUPPORTED_DEVICE = 8
ATTN_ERR_WORKSPACE = 9

ATTN_KERNEL_AUTO = -1      # attn_fwd_variant: the kernel attn_fwd would run
ATTN_KERNEL_ONE_TILE = 0   # units of 128 query rows
ATTN_KERNEL_TWO_TILE = 1   # units of two 128-row query tiles
ATTN_V_ROWS = 0        # E4M3 V as [B, H, Sk, D]
ATTN_V_TRANSPOSED = 1  # E4M3 V as [B, H, D, Sk]

#: Functions declared in include/attn.h, with their ctypes signatures.
SIGNATURES = {
    "attn_fwd": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "attn_fwd_variant": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                        ctypes.c_void_p]),
    "attn_fwd_fp8": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_float,
                                    ctypes.c_float, ctypes.c_float, ctypes.c_void_p]),
    "attn_fwd_fp8_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_float,
                                       ctypes.c_float, ctypes.c_float, ctypes.c_int, ctypes.c_void_p]),
    "attn_fwd_fp8_variant": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_void_p,
                                            ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_void_p]),
    "attn_fwd_varlen": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                       ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "attn_fwd_varlen_variant": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                               ctypes.c_void_p]),
    "attn_fwd_paged": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_void_p]),
    "attn_fwd_paged_variant": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                              ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]),
    "attn_fwd_splitkv_workspace_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                          ctypes.c_int]),
    "attn_fwd_splitkv_suggest_splits": (ctypes.c_int, [ctypes.c_int] * 5),
    "attn_fwd_splitkv": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "attn_fwd_splitkv_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_void_p,
                                                ctypes.c_int, ctypes.c_void_p]),
    "attn_lse_merge": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_void_p]),
    "attn_bwd_workspace_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "attn_bwd": (ctypes.c_int, [ctypes.c_void_p] * 9 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int,
                                                                          ctypes.c_void_p, ctypes.c_void_p,
                                                                          ctypes.c_size_t, ctypes.c_void_p]),
    "attn_get_error_string": (ctypes.c_char_p, [ctypes.c_int]),
    "attn_check_device_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]),
    "attn_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_int64, ctypes.c_void_p]),
    "attn_selftest_launch_floor": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "attn_selftest_fwd_abort": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int,
                                                                                          ctypes.c_void_p, ctypes.c_int,
                                                                                          ctypes.c_int, ctypes.c_int64,
                                                                                          ctypes.c_void_p]),
    "attn_fwd_kernel_choice": (ctypes.c_int, [ctypes.c_int] * 7),
    "attn_fwd_fp8_kernel_choice": (ctypes.c_int, [ctypes.c_int] * 7),
    "attn_fwd_pair_schedule": (ctypes.c_int64, [ctypes.c_int] * 6 + [ctypes.c_void_p, ctypes.c_int64]),
    "attn_abi_version": (ctypes.c_int, []),
}


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {attn_get_error_string(status)} (status {status})" if what
                         else f"{attn_get_error_string(status)} (status {status})")


def library_path() -> str:
    return _LIB_PATH


def lib():
    """Load ``libattn.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "`python -m exact_attention_86_gb300.build` (needs nvcc)")
        handle = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


# ----------------------------------------------------------------- raw C ABI

def attn_fwd(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, Sq: int, Sk: int, D: int,
             scale: float, causal: int, kv_lens: Optional[int], stream: Optional[int]) -> int:
    return lib().attn_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, scale, int(causal), kv_lens, stream)


def attn_fwd_variant(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, Sq: int, Sk: int, D: int,
                     scale: float, causal: int, kv_lens: Optional[int], kernel: int, stream: Optional[int]) -> int:
    return lib().attn_fwd_variant(q, k, v, o, lse, B, H, Sq, Sk, D, scale, int(causal), kv_lens, kernel, stream)


def attn_fwd_fp8(q: int, k: int, v_t: int, o: int, lse: int, B: int, H: int, Sq: int, Sk: int, D: int,
                 scale: float, causal: int, kv_lens: Optional[int], q_descale: float, k_descale: float,
                 v_descale: float, stream: Optional[int]) -> int:
    return lib().attn_fwd_fp8(q, k, v_t, o, lse, B, H, Sq, Sk, D, scale, int(causal), kv_lens, q_descale, k_descale,
                              v_descale, stream)


def attn_fwd_fp8_variant(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, Sq: int, Sk: int, D: int,
                         scale: float, causal: int, kv_lens: Optional[int], q_descale: float, k_descale: float,
                         v_descale: float, v_layout: int, kernel: int, stream: Optional[int]) -> int:
    return lib().attn_fwd_fp8_variant(q, k, v, o, lse, B, H, Sq, Sk, D, scale, int(causal), kv_lens, q_descale,
                                      k_descale, v_descale, v_layout, kernel, stream)


def attn_fwd_fp8_ex(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, Sq: int, Sk: int, D: int,
                    scale: float, causal: int, kv_lens: Optional[int], q_descale: float, k_descale: float,
                    v_descale: float, v_layout: int, stream: Optional[int]) -> int:
    return lib().attn_fwd_fp8_ex(q, k, v, o, lse, B, H, Sq, Sk, D, scale, int(causal), kv_lens, q_descale,
                                 k_descale, v_descale, v_layout, stream)


def attn_fwd_varlen(q: int, k: int, v: int, o: int, lse: int, cu_q: int, cu_k: int, batch: int,
                    max_seqlen_q: int, total_q: int, total_k: int, H: int, D: int, scale: float, causal: int,
                    tile_counter: Optional[int], stream: Optional[int]) -> int:
    return lib().attn_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, batch, max_seqlen_q, total_q, total_k, H, D, scale,
                                 int(causal), tile_counter, stream)


def attn_fwd_varlen_variant(q: int, k: int, v: int, o: int, lse: int, cu_q: int, cu_k: int, batch: int,
                            max_seqlen_q: int, total_q: int, total_k: int, H: int, D: int, scale: float, causal: int,
                            tile_counter: Optional[int], kernel: int, stream: Optional[int]) -> int:
    return lib().attn_fwd_varlen_variant(q, k, v, o, lse, cu_q, cu_k, batch, max_seqlen_q, total_q, total_k, H, D,
                                         scale, int(causal), tile_counter, kernel, stream)


def attn_fwd_paged(q: int, k_cache: int, v_cache: int, o: int, lse: int, cu_q: int, seqlens_k: int,
                   block_table: int, batch: int, max_seqlen_q: int, total_q: int, num_pages: int, page_size: int,
                   max_pages_per_seq: int, H: int, D: int, scale: float, causal: int, tile_counter: Optional[int],
                   stream: Optional[int]) -> int:
    return lib().attn_fwd_paged(q, k_cache, v_cache, o, lse, cu_q, seqlens_k, block_table, batch, max_seqlen_q,
                                total_q, num_pages, page_size, max_pages_per_seq, H, D, scale, int(causal),
                                tile_counter, stream)


def attn_fwd_paged_variant(q: int, k_cache: int, v_cache: int, o: int, lse: int, cu_q: int, seqlens_k: int,
                           block_table: int, batch: int, max_seqlen_q: int, total_q: int, num_pages: int,
                           page_size: int, max_pages_per_seq: int, H: int, D: int, scale: float, causal: int,
                           tile_counter: Optional[int], kernel: int, stream: Optional[int]) -> int:
    return lib().attn_fwd_paged_variant(q, k_cache, v_cache, o, lse, cu_q, seqlens_k, block_table, batch,
                                        max_seqlen_q, total_q, num_pages, page_size, max_pages_per_seq, H, D, scale,
                                        int(causal), tile_counter, kernel, stream)


def attn_fwd_splitkv_workspace_size(B: int, H: int, Sq: int, D: int, num_splits: int) -> int:
    return lib().attn_fwd_splitkv_workspace_size(B, H, Sq, D, num_splits)


def attn_fwd_splitkv_suggest_splits(B: int, H: int, Sq: int, Sk: int, num_sms: int) -> int:
    return lib().attn_fwd_splitkv_suggest_splits(B, H, Sq, Sk, num_sms)


def attn_fwd_splitkv(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, Sq: int, Sk: int, D: int,
                     scale: float, causal: int, kv_lens: Optional[int], num_splits: int, workspace: int,
                     workspace_bytes: int, stream: Optional[int]) -> int:
    return lib().attn_fwd_splitkv(q, k, v, o, lse, B, H, Sq, Sk, D, scale, int(causal), kv_lens, num_splits,
                                  workspace, workspace_bytes, stream)


def attn_fwd_splitkv_noalloc(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, Sq: int, Sk: int, D: int,
                             scale: float, causal: int, kv_lens: Optional[int], num_splits: int,
                             stream: Optional[int]) -> int:
    return lib().attn_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, Sq, Sk, D, scale, int(causal), kv_lens, num_splits,
                                          stream)


def attn_lse_merge(o_parts: int, lse_parts: int, num_parts: int, o: int, lse: int, rows: int, D: int,
                   stream: Optional[int]) -> int:
    return lib().attn_lse_merge(o_parts, lse_parts, num_parts, o, lse, rows, D, stream)


def attn_bwd_workspace_size(B: int, H: int, Sq: int) -> int:
    return lib().attn_bwd_workspace_size(B, H, Sq)


def attn_bwd(q: int, k: int, v: int, o: int, dout: int, lse: int, dq: int, dk: int, dv: int, B: int, H: int, Sq: int,
             Sk: int, D: int, scale: float, causal: int, kv_lens: Optional[int], workspace: Optional[int],
             workspace_bytes: int, stream: Optional[int]) -> int:
    return lib().attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, Sq, Sk, D, scale, int(causal), kv_lens, workspace,
                          workspace_bytes, stream)


def attn_get_error_string(status: int) -> str:
    return lib().attn_get_error_string(status).decode()


def attn_check_device_status(stream: Optional[int] = None) -> Tuple[int, int]:
    site = ctypes.c_uint32(0)
    st = lib().attn_check_device_status(stream, ctypes.byref(site))
    return st, site.value


def attn_selftest_wait_timeout(limit_ns: int, stream: Optional[int] = None) -> int:
    return lib().attn_selftest_wait_timeout(limit_ns, stream)


def attn_selftest_fwd_abort(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, Sq: int, Sk: int, D: int,
                            scale: float, causal: int, kv_lens: Optional[int], kernel: int, skip_fill: int,
                            limit_ns: int, stream: Optional[int] = None) -> int:
    return lib().attn_selftest_fwd_abort(q, k, v, o, lse, B, H, Sq, Sk, D, scale, int(causal), kv_lens, kernel,
                                         skip_fill, limit_ns, stream)


def attn_selftest_launch_floor(grid: int, D: int, mode: int, stream: Optional[int] = None) -> int:
    return lib().attn_selftest_launch_floor(grid, D, mode, stream)


def attn_fwd_kernel_choice(B: int, H: int, Sq: int, Sk: int, D: int, causal: int, num_sms: int) -> int:
    return lib().attn_fwd_kernel_choice(B, H, Sq, Sk, D, int(causal), num_sms)


def attn_fwd_fp8_kernel_choice(B: int, H: int, Sq: int, Sk: int, D: int, causal: int, num_sms: int) -> int:
    return lib().attn_fwd_fp8_kernel_choice(B, H, Sq, Sk, D, int(causal), num_sms)


def attn_fwd_pair_schedule(B: int, H: int, Sq: int, Sk: int, head_group: int, grid: int, max_units: int = 4096):
    """The static deal of a causal batch's two-tile units: a bytes object whose
    entry t is the block that runs unit t, or None when the library declines
    (too many units or an argument out of range)."""
    buf = (ctypes.c_uint8 * max(max_units, 1))()
    n = lib().attn_fwd_pair_schedule(B, H, Sq, Sk, head_group, grid, buf, max_units)
    return None if n < 0 else bytes(buf[:n])


def attn_abi_version() -> int:
    return lib().attn_abi_version()


# -------------------------------------------------------------- torch facing

def _check_qkv(q, k, v, kv_lens):
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-d bf16 CUDA tensor")
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    if tuple(k.shape) != (B, H, Sk, D) or tuple(v.shape) != (B, H, Sk, D):
        raise ValueError("k and v must be [B, H, Sk, D] with q's B, H, D")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k, v must be on one device")
    kv_ptr = None
    if kv_lens is not None:
        if kv_lens.dtype != torch.int32 or kv_lens.device != q.device or kv_lens.numel() != B \
                or not kv_lens.is_contiguous():
            raise ValueError("kv_lens must be a contiguous int32 tensor [B] on q's device")
        kv_ptr = kv_lens.data_ptr()
    return B, H, Sq, Sk, D, kv_ptr


def _outputs(out, lse, o_shape, lse_shape, device):
    """The caller's output tensors (checked) or new ones."""
    import torch

    if out is None:
        out = torch.empty(o_shape, dtype=torch.bfloat16, device=device)
    elif out.dtype != torch.bfloat16 or out.device != device or not out.is_contiguous() \
            or tuple(out.shape) != tuple(o_shape):
        raise ValueError(f"out must be a contiguous bf16 tensor {tuple(o_shape)} on the inputs' device")
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=device)
    elif lse.dtype != torch.float32 or lse.device != device or not lse.is_contiguous() \
            or tuple(lse.shape) != tuple(lse_shape):
        raise ValueError(f"lse must be a contiguous fp32 tensor {tuple(lse_shape)} on the inputs' device")
    return out, lse


MAX_SPLITS = 128  # attn_fwd_splitkv accepts 1 .. 128 key ranges


def suggest_num_splits(B: int, H: int, Sq: int, Sk: int, num_sms: int) -> int:
    """Key ranges for attn_fwd_splitkv on a GPU with num_sms SMs (the
    library's attn_fwd_splitkv_suggest_splits: within one wave of SMs, equal
    ranges preferred)."""
    return attn_fwd_splitkv_suggest_splits(B, H, Sq, Sk, num_sms)


def forward_splitkv(q, k, v, num_splits: Optional[int] = None, scale: Optional[float] = None,
                    causal: bool = False, kv_lens=None, workspace=None):
    """Split-KV forward on torch CUDA tensors (see ``forward``).
    ``num_splits`` None picks ``suggest_num_splits`` for the device's SM
    count.  ``workspace`` (a CUDA tensor of at least
    ``attn_fwd_splitkv_workspace_size`` bytes) is allocated with torch when not
    given."""
    import torch

    B, H, Sq, Sk, D, kv_ptr = _check_qkv(q, k, v, kv_lens)
    if num_splits is None:
        num_splits = suggest_num_splits(B, H, Sq, Sk, torch.cuda.get_device_properties(q.device).multi_processor_count)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = torch.empty((B, H, Sq, D), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    need = attn_fwd_splitkv_workspace_size(B, H, Sq, D, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        st = attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                              B, H, Sq, Sk, D, float(scale), int(bool(causal)), kv_ptr, num_splits,
                              workspace.data_ptr(), workspace.numel() * workspace.element_size(), stream)
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_splitkv")
    return out, lse


def forward_fp8(q8, k8, v8, q_descale: float = 1.0, k_descale: float = 1.0, v_descale: float = 1.0,
                scale: Optional[float] = None, causal: bool = False, kv_lens=None, out=None, lse=None,
                v_layout: int = ATTN_V_TRANSPOSED, kernel: int = ATTN_KERNEL_AUTO):
    """FP8 forward on torch CUDA tensors of E4M3 codes (``torch.uint8`` or
    ``torch.float8_e4m3fn``): ``q8 [B,H,Sq,D]``, ``k8 [B,H,Sk,D]`` and ``v8``,
    which is ``[B,H,D,Sk]`` (V transposed) with ``v_layout=ATTN_V_TRANSPOSED``
    (the default) or ``[B,H,Sk,D]`` with ``v_layout=ATTN_V_ROWS``.  ``kernel``
    as for ``forward``.  Returns ``(o bf16 [B,H,Sq,D], lse fp32 [B,H,Sq])``,
    written into ``out`` / ``lse`` when given."""
    import torch

    for name, t in (("q8", q8), ("k8", k8), ("v8", v8)):
        if t.element_size() != 1 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-d CUDA tensor of 1-byte E4M3 codes")
    B, H, Sq, D = q8.shape
    Sk = k8.shape[2]
    v_shape = (B, H, Sk, D) if v_layout == ATTN_V_ROWS else (B, H, D, Sk)
    if tuple(k8.shape) != (B, H, Sk, D) or tuple(v8.shape) != v_shape:
        raise ValueError(f"k8 must be [B,H,Sk,D] and v8 {list(v_shape)}")
    if kv_lens is not None and (kv_lens.dtype != torch.int32 or kv_lens.device != q8.device):
        raise ValueError("kv_lens must be int32 on q's device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out, lse = _outputs(out, lse, (B, H, Sq, D), (B, H, Sq), q8.device)
    with torch.cuda.device(q8.device):
        stream = torch.cuda.current_stream(q8.device).cuda_stream
        st = attn_fwd_fp8_variant(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), out.data_ptr(), lse.data_ptr(), B,
                                  H, Sq, Sk, D, float(scale), int(bool(causal)),
                                  None if kv_lens is None else kv_lens.data_ptr(), float(q_descale),
                                  float(k_descale), float(v_descale), int(v_layout), int(kernel), stream)
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_fp8")
    return out, lse


_counters = {}


def tile_counter(device, stream: int):
    """A zeroed device uint32[2] for dynamic scheduling, one per (device,
    stream); every launch leaves it zero again, so calls on one stream can
    share it."""
    import torch

    key = (str(device), int(stream or 0))
    t = _counters.get(key)
    if t is None:
        t = torch.zeros(2, dtype=torch.int32, device=device)
        _counters[key] = t
    return t


def forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, scale: Optional[float] = None,
                   causal: bool = False, dynamic: bool = True, out=None, lse=None, kernel: int = ATTN_KERNEL_AUTO):
    """Packed variable-length forward on torch CUDA tensors: ``q [total_q, H, D]``,
    ``k``/``v [total_k, H, D]`` bf16, ``cu_seqlens_q``/``cu_seqlens_k`` int32
    ``[batch + 1]`` on the same device.  ``kernel`` as for ``forward``.
    Returns ``(o [total_q, H, D], lse [H, total_q])``, written into ``out`` /
    ``lse`` when given."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 3:
            raise ValueError(f"{name} must be a contiguous 3-d bf16 CUDA tensor")
    total_q, H, D = q.shape
    total_k = k.shape[0]
    if tuple(k.shape) != (total_k, H, D) or tuple(v.shape) != (total_k, H, D):
        raise ValueError("k and v must be [total_k, H, D] with q's H, D")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if t.dtype != torch.int32 or t.device != q.device or not t.is_contiguous() or t.dim() != 1:
            raise ValueError(f"{name} must be a contiguous int32 tensor on q's device")
    batch = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != batch + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out, lse = _outputs(out, lse, (total_q, H, D), (H, total_q), q.device)
    with torch.cuda.device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        counter = tile_counter(q.device, stream).data_ptr() if dynamic else None
        st = attn_fwd_varlen_variant(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                     cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), batch, int(max_seqlen_q),
                                     total_q, total_k, H, D, float(scale), int(bool(causal)), counter, int(kernel),
                                     stream)
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_varlen")
    return out, lse


def forward_paged(q, k_cache, v_cache, cu_seqlens_q, seqlens_k, block_table, max_seqlen_q: int,
                  scale: Optional[float] = None, causal: bool = False, dynamic: bool = True, out=None, lse=None,
                  kernel: int = ATTN_KERNEL_AUTO):
    """Packed queries ``q [total_q, H, D]`` against a paged KV cache
    ``k_cache``/``v_cache [num_pages, page_size, H, D]`` (bf16 CUDA tensors);
    ``cu_seqlens_q`` int32 ``[batch + 1]``, ``seqlens_k`` int32 ``[batch]``,
    ``block_table`` int32 ``[batch, max_pages_per_seq]`` on the same device.
    Returns ``(o [total_q, H, D], lse [H, total_q])``, written into ``out`` /
    ``lse`` when given."""
    import torch

    if q.dtype != torch.bfloat16 or not q.is_cuda or not q.is_contiguous() or q.dim() != 3:
        raise ValueError("q must be a contiguous 3-d bf16 CUDA tensor")
    total_q, H, D = q.shape
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        if t.dtype != torch.bfloat16 or t.device != q.device or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-d bf16 tensor on q's device")
    num_pages, page_size = k_cache.shape[0], k_cache.shape[1]
    if tuple(k_cache.shape) != (num_pages, page_size, H, D) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache must be [num_pages, page_size, H, D] with q's H, D")
    for name, t, dim in (("cu_seqlens_q", cu_seqlens_q, 1), ("seqlens_k", seqlens_k, 1),
                         ("block_table", block_table, 2)):
        if t.dtype != torch.int32 or t.device != q.device or not t.is_contiguous() or t.dim() != dim:
            raise ValueError(f"{name} must be a contiguous {dim}-d int32 tensor on q's device")
    batch = cu_seqlens_q.numel() - 1
    if seqlens_k.numel() != batch or block_table.shape[0] != batch:
        raise ValueError("seqlens_k and block_table must have one entry (row) per sequence")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out, lse = _outputs(out, lse, (total_q, H, D), (H, total_q), q.device)
    with torch.cuda.device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        counter = tile_counter(q.device, stream).data_ptr() if dynamic else None
        st = attn_fwd_paged_variant(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                                    lse.data_ptr(), cu_seqlens_q.data_ptr(), seqlens_k.data_ptr(),
                                    block_table.data_ptr(), batch, int(max_seqlen_q), total_q, num_pages, page_size,
                                    block_table.shape[1], H, D, float(scale), int(bool(causal)), counter,
                                    int(kernel), stream)
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_paged")
    return out, lse


def backward(q, k, v, o, lse, dout, scale: Optional[float] = None, causal: bool = False, kv_lens=None):
    """Gradients ``(dq, dk, dv)`` (bf16, shaped like q, k, v) of the forward's
    ``o`` for the upstream gradient ``dout``; ``o`` and ``lse`` are the
    forward's outputs for the same arguments."""
    import torch

    _check_qkv(q, k, v, kv_lens)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    for name, t in (("o", o), ("dout", dout)):
        if t.dtype != torch.bfloat16 or t.device != q.device or not t.is_contiguous() or tuple(t.shape) != tuple(q.shape):
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    if lse.dtype != torch.float32 or lse.device != q.device or tuple(lse.shape) != (B, H, Sq):
        raise ValueError("lse must be fp32 [B, H, Sq] on q's device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    ws_bytes = attn_bwd_workspace_size(B, H, Sq)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        st = attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                      dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Sq, Sk, D, float(scale), int(bool(causal)),
                      None if kv_lens is None else kv_lens.data_ptr(), ws.data_ptr(), ws.numel(), stream)
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")
    return dq, dk, dv


def lse_merge(o_parts, lse_parts):
    """Merge ``o_parts`` (fp32 ``[n, rows, D]``) and ``lse_parts`` (fp32 ``[n, rows]``)
    CUDA tensors into ``(o bf16 [rows, D], lse fp32 [rows])``."""
    import torch

    n, rows, D = o_parts.shape
    out = torch.empty((rows, D), dtype=torch.bfloat16, device=o_parts.device)
    lse = torch.empty((rows,), dtype=torch.float32, device=o_parts.device)
    with torch.cuda.device(o_parts.device):
        stream = torch.cuda.current_stream(o_parts.device).cuda_stream
        st = attn_lse_merge(o_parts.data_ptr(), lse_parts.data_ptr(), n, out.data_ptr(), lse.data_ptr(), rows, D,
                            stream)
    if st != ATTN_OK:
        raise AttnError(st, "attn_lse_merge")
    return out, lse


def forward(q, k, v, scale: Optional[float] = None, causal: bool = False, kv_lens=None,
            out=None, lse=None, kernel: int = ATTN_KERNEL_AUTO):
    """Fused attention forward on torch CUDA tensors.

    ``q [B,H,Sq,D]``, ``k``/``v [B,H,Sk,D]``: bf16, contiguous, same device.
    ``kv_lens``: ``None`` or an int32 CUDA tensor ``[B]``.  ``scale`` defaults to
    ``1/sqrt(D)``.  ``kernel``: ``ATTN_KERNEL_AUTO`` (``attn_fwd``) or a kernel
    forced through ``attn_fwd_variant``.  Returns ``(o bf16 [B,H,Sq,D], lse
    fp32 [B,H,Sq])``.  The call is asynchronous on the current stream."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-d bf16 CUDA tensor")
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    if tuple(k.shape) != (B, H, Sk, D) or tuple(v.shape) != (B, H, Sk, D):
        raise ValueError("k and v must be [B, H, Sk, D] with q's B, H, D")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k, v must be on one device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    kv_ptr = None
    if kv_lens is not None:
        if kv_lens.dtype != torch.int32 or kv_lens.device != q.device or kv_lens.numel() != B \
                or not kv_lens.is_contiguous():
            raise ValueError("kv_lens must be a contiguous int32 tensor [B] on q's device")
        kv_ptr = kv_lens.data_ptr()
    out, lse = _outputs(out, lse, (B, H, Sq, D), (B, H, Sq), q.device)
    with torch.cuda.device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        if kernel == ATTN_KERNEL_AUTO:
            st = attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                          B, H, Sq, Sk, D, float(scale), int(bool(causal)), kv_ptr, stream)
        else:
            st = attn_fwd_variant(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                  B, H, Sq, Sk, D, float(scale), int(bool(causal)), kv_ptr, int(kernel), stream)
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd" if kernel == ATTN_KERNEL_AUTO else "attn_fwd_variant")
    return out, lse
