"""exact_io_aware_gb300 — exact tiled softmax attention on GB300, Python binding.

A thin ctypes layer over the C ABI in ``include/exactattn.h`` (``lib/libexactattn.so``):
it checks tensor shapes, allocates outputs with PyTorch and passes raw device pointers and
the current CUDA stream.  All arithmetic runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback, and every entry point raises if the library is not built.

    o, lse = attn_fwd(q, k, v, c, mask="causal")
    o, lse = attn_fwd_split(q, k, v, c, mask="causal")   # key shares + merge (few heads)
    dq, dk, dv = attn_bwd(q, k, v, o, lse, do, c, mask="causal")
    y = attention(q, k, v, c, mask="causal")      # autograd-aware wrapper
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "attn_fwd_dropout", "attn_bwd_dropout", "attn_fwd_kv", "attn_fwd_kv_split_count",
    "attn_fwd_fp8", "attn_fp8_quantize", "attn_fwd_fp8_blocks", "attn_fwd_vdim", "attn_bwd_vdim",
    "AttnError", "ATTN_OK", "ATTN_WARN_EMPTY_ROW", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED",
    "ATTN_ERR_ALIGNMENT", "ATTN_ERR_WORKSPACE", "ATTN_ERR_CUDA", "ATTN_ERR_DEVICE_TIMEOUT",
    "library_path", "load", "attn_fwd", "attn_bwd", "attn_bwd_workspace_bytes",
    "attn_device_status", "attn_last_error", "attention", "attn_bwd_noalloc",
    "attn_selftest_wait_timeout", "attn_fwd_split", "attn_fwd_split_count",
    "attn_fwd_split_workspace_bytes", "attn_merge", "attn_selftest_exp2",
    "attn_debug_set_ring_stages",
]


ATTN_OK = 0
ATTN_WARN_EMPTY_ROW = 1
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_ALIGNMENT = -3
ATTN_ERR_WORKSPACE = -4
ATTN_ERR_CUDA = -5
ATTN_ERR_DEVICE_TIMEOUT = -6

DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
MASK_CODE = {"none": 0, "causal": 1, "bitmap": 2}

_lib = None


class AttnError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"exactattn error {code}: {message}")
        self.code = code


def library_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libexactattn.so")


def load():
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with exact_io_aware_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.attn_fwd.argtypes = [i32, i32, i32, i32, i32, f32, vp, vp, vp, i32, vp, i64, i64, i32,
                             vp, vp, vp]
    lib.attn_fwd.restype = i32
    lib.attn_bwd_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    lib.attn_bwd_workspace_bytes.restype = sz
    lib.attn_bwd.argtypes = [i32, i32, i32, i32, i32, f32, vp, vp, vp, vp, vp, vp, i32, vp, i64,
                             i64, i32, vp, vp, vp, vp, sz, vp]
    lib.attn_bwd.restype = i32
    lib.attn_device_status.argtypes = [vp]
    lib.attn_device_status.restype = i32
    lib.attn_last_error.argtypes = []
    lib.attn_last_error.restype = ctypes.c_char_p
    lib.attn_fwd_split.argtypes = [i32, i32, i32, i32, i32, f32, vp, vp, vp, i32, vp, i64, i64,
                                   i32, i32, vp, vp, vp, sz, vp]
    lib.attn_fwd_split.restype = i32
    lib.attn_fwd_split_count.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.attn_fwd_split_count.restype = i32
    lib.attn_fwd_split_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.attn_fwd_split_workspace_bytes.restype = sz
    lib.attn_merge.argtypes = [i32, i32, i64, i32, vp, vp, vp, vp, vp]
    lib.attn_merge.restype = i32
    lib.attn_fwd_kv.argtypes = [i32, i32, i32, i32, i32, i32, f32, vp, vp, vp, i32, vp, i64, i64,
                                i32, i32, vp, vp, vp, sz, vp]
    lib.attn_fwd_kv.restype = i32
    lib.attn_fwd_kv_split_count.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.attn_fwd_kv_split_count.restype = i32
    lib.attn_fwd_fp8.argtypes = [i32, i32, i32, i32, f32, vp, vp, vp, f32, f32, f32, i32, vp, i64,
                                 i64, vp, vp, vp]
    lib.attn_fwd_fp8.restype = i32
    lib.attn_fwd_fp8_blocks.argtypes = [i32, i32, i32, i32, f32, vp, vp, vp, vp, vp, vp, i32, vp,
                                        i64, i64, vp, vp, vp]
    lib.attn_fwd_fp8_blocks.restype = i32
    lib.attn_fp8_quantize.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      vp, vp]
    lib.attn_fp8_quantize.restype = i32
    lib.attn_fwd_vdim.argtypes = [i32, i32, i32, i32, i32, i32, f32, vp, vp, vp, i32, vp, i64, i64,
                                  i32, f32, ctypes.c_uint64, vp, vp, vp]
    lib.attn_fwd_vdim.restype = i32
    lib.attn_bwd_vdim.argtypes = [i32, i32, i32, i32, i32, i32, f32, vp, vp, vp, vp, vp, vp, i32,
                                  vp, i64, i64, i32, f32, ctypes.c_uint64, vp, vp, vp, vp, sz, vp]
    lib.attn_bwd_vdim.restype = i32
    u64 = ctypes.c_uint64
    lib.attn_fwd_dropout.argtypes = [i32, i32, i32, i32, i32, f32, vp, vp, vp, i32, vp, i64, i64,
                                     i32, f32, u64, vp, vp, vp]
    lib.attn_fwd_dropout.restype = i32
    lib.attn_bwd_dropout.argtypes = [i32, i32, i32, i32, i32, f32, vp, vp, vp, vp, vp, vp, i32,
                                     vp, i64, i64, i32, f32, u64, vp, vp, vp, vp, sz, vp]
    lib.attn_bwd_dropout.restype = i32
    lib.attn_selftest_exp2.argtypes = [vp, vp, vp, i64, vp]
    lib.attn_debug_set_ring_stages.argtypes = [i32]
    lib.attn_debug_set_ring_stages.restype = i32
    lib.attn_selftest_exp2.restype = i32
    _lib = lib
    return lib


def attn_last_error() -> str:
    return load().attn_last_error().decode()


def _check(rc: int):
    if rc < 0:
        raise AttnError(rc, attn_last_error())
    return rc


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _shape(q, k, v):
    if q.dim() != 4:
        raise ValueError("q, k, v must be [B, H, n, d]")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k and v must have the same shape (n_q = n_k, v = d)")
    if q.dtype not in DTYPE_CODE or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype among float32, float16, bfloat16")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    return q.shape


def _shape_v(q, k, v):
    """(B, H, n, d, v_dim): q, k [B,H,n,d] and v [B,H,n,v_dim] (v_dim may differ from d)."""
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("q, k must be [B,H,n,d] and v [B,H,n,v]")
    if q.dtype not in DTYPE_CODE or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype among float32, float16, bfloat16")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    return (*q.shape, v.shape[3])


def _mask_args(mask, mask_bits, mask_head_stride_words):
    kind = MASK_CODE[mask]
    if kind != 2:
        return kind, None, 0, 0
    if mask_bits is None or not mask_bits.is_cuda or not mask_bits.is_contiguous():
        raise ValueError("bitmap mask needs a contiguous CUDA int32 tensor [..., n, row_words]")
    if mask_bits.dtype not in (torch.int32, torch.uint32):
        raise ValueError("mask_bits must hold 32-bit words")
    return kind, mask_bits, int(mask_bits.shape[-1]), int(mask_head_stride_words)


def attn_fwd(q, k, v, c, mask="none", mask_bits=None, mask_head_stride_words=0, kv_block=0,
             o=None, lse=None, stream=None, dropout_p=0.0, seed=0):
    """Forward pass; returns (o [B,H,n,v], lse [B,H,n] float32).  dropout_p > 0 drops
    probabilities with the library's replayable mask for ``seed`` (attn_fwd_dropout).  v may
    be narrower or wider than q and k (attn_fwd_vdim)."""
    B, H, n, d, v_dim = _shape_v(q, k, v)
    kind, bits, row_words, hs = _mask_args(mask, mask_bits, mask_head_stride_words)
    if o is None:
        o = torch.empty_like(v)
    if lse is None:
        lse = torch.empty((B, H, n), dtype=torch.float32, device=q.device)
    lib = load()
    if v_dim != d:
        _check(lib.attn_fwd_vdim(DTYPE_CODE[q.dtype], B, H, n, d, v_dim, float(c), _ptr(q),
                                 _ptr(k), _ptr(v), kind, _ptr(bits), row_words, hs,
                                 int(kv_block), float(dropout_p), int(seed) & 0xFFFFFFFFFFFFFFFF,
                                 _ptr(o), _ptr(lse), _stream_ptr(stream)))
        return o, lse
    if dropout_p:
        _check(lib.attn_fwd_dropout(DTYPE_CODE[q.dtype], B, H, n, d, float(c), _ptr(q), _ptr(k),
                                    _ptr(v), kind, _ptr(bits), row_words, hs, int(kv_block),
                                    float(dropout_p), int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(o),
                                    _ptr(lse), _stream_ptr(stream)))
        return o, lse
    _check(lib.attn_fwd(DTYPE_CODE[q.dtype], B, H, n, d, float(c), _ptr(q), _ptr(k), _ptr(v),
                        kind, _ptr(bits), row_words, hs, int(kv_block), _ptr(o), _ptr(lse),
                        _stream_ptr(stream)))
    return o, lse


def attn_fwd_split_count(dtype, B, H, n, d, kv_block=0) -> int:
    """Key shares attn_fwd_split uses with num_splits=0 on the current device."""
    code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load().attn_fwd_split_count(code, B, H, n, d, int(kv_block)))


def attn_fwd_split_workspace_bytes(dtype, B, H, n, d, num_splits) -> int:
    code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load().attn_fwd_split_workspace_bytes(code, B, H, n, d, int(num_splits)))


def attn_fwd_split(q, k, v, c, mask="none", mask_bits=None, mask_head_stride_words=0,
                   kv_block=0, num_splits=0, o=None, lse=None, workspace=None, stream=None):
    """Forward pass over num_splits key shares merged into (o, lse); 0 = library choice."""
    B, H, n, d = _shape(q, k, v)
    kind, bits, row_words, hs = _mask_args(mask, mask_bits, mask_head_stride_words)
    splits = int(num_splits) or attn_fwd_split_count(q.dtype, B, H, n, d, kv_block)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, n), dtype=torch.float32, device=q.device)
    need = attn_fwd_split_workspace_bytes(q.dtype, B, H, n, d, splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(load().attn_fwd_split(DTYPE_CODE[q.dtype], B, H, n, d, float(c), _ptr(q), _ptr(k),
                                 _ptr(v), kind, _ptr(bits), row_words, hs, int(kv_block), splits,
                                 _ptr(o), _ptr(lse), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(),
                                 _stream_ptr(stream)))
    return o, lse


def attn_fwd_kv_split_count(dtype, B, H, n_q, n_kv, d, kv_block=0) -> int:
    """Key shares attn_fwd_kv uses with num_splits=0 on the current device."""
    code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load().attn_fwd_kv_split_count(code, B, H, n_q, n_kv, d, int(kv_block)))


def attn_fwd_kv(q, k, v, c, mask="none", mask_bits=None, mask_head_stride_words=0, kv_block=0,
                num_splits=0, o=None, lse=None, workspace=None, stream=None):
    """Forward of q [B,H,n_q,d] against a key/value cache k, v [B,H,n_kv,d] (queries at the end
    of the sequence under the causal mask); returns (o [B,H,n_q,d], lse [B,H,n_q])."""
    if q.dim() != 4 or k.shape != v.shape or k.dim() != 4:
        raise ValueError("q must be [B,H,n_q,d] and k, v [B,H,n_kv,d]")
    B, H, n_q, d = q.shape
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != d:
        raise ValueError("q, k, v must agree on B, H and d")
    n_kv = k.shape[2]
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype or t.dtype not in DTYPE_CODE:
            raise ValueError("q, k, v must be contiguous CUDA tensors of one supported dtype")
    kind, bits, row_words, hs = _mask_args(mask, mask_bits, mask_head_stride_words)
    splits = int(num_splits) or attn_fwd_kv_split_count(q.dtype, B, H, n_q, n_kv, d, kv_block)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, n_q), dtype=torch.float32, device=q.device)
    need = attn_fwd_split_workspace_bytes(q.dtype, B, H, n_q, d, splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(load().attn_fwd_kv(DTYPE_CODE[q.dtype], B, H, n_q, n_kv, d, float(c), _ptr(q), _ptr(k),
                              _ptr(v), kind, _ptr(bits), row_words, hs, int(kv_block), splits,
                              _ptr(o), _ptr(lse), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream_ptr(stream)))
    return o, lse


def _fp8_bytes(t, name):
    if t.dtype not in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        raise ValueError(f"{name} must hold E4M3 values (torch.float8_e4m3fn or uint8)")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t


def attn_fwd_fp8(q8, k8, vt8, c, q_scale, k_scale, v_scale, mask="none", mask_bits=None,
                 mask_head_stride_words=0, o=None, lse=None, stream=None):
    """FP8 forward: q8, k8 E4M3 [B,H,n,d], vt8 E4M3 [B,H,d,n] (V transposed), one scale per
    tensor; returns (o bfloat16 [B,H,n,d], lse float32 [B,H,n])."""
    q8, k8, vt8 = (_fp8_bytes(t, nm) for t, nm in ((q8, "q8"), (k8, "k8"), (vt8, "vt8")))
    if q8.dim() != 4 or k8.shape != q8.shape:
        raise ValueError("q8 and k8 must be [B,H,n,d]")
    B, H, n, d = q8.shape
    if tuple(vt8.shape) != (B, H, d, n):
        raise ValueError("vt8 must be [B,H,d,n] (V transposed)")
    kind, bits, row_words, hs = _mask_args(mask, mask_bits, mask_head_stride_words)
    if o is None:
        o = torch.empty((B, H, n, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, n), dtype=torch.float32, device=q8.device)
    _check(load().attn_fwd_fp8(B, H, n, d, float(c), _ptr(q8), _ptr(k8), _ptr(vt8),
                               float(q_scale), float(k_scale), float(v_scale), kind, _ptr(bits),
                               row_words, hs, _ptr(o), _ptr(lse), _stream_ptr(stream)))
    return o, lse


def attn_fwd_vdim(q, k, v, c, **kw):
    """Forward with v [B,H,n,v] of its own width (the same call as attn_fwd)."""
    return attn_fwd(q, k, v, c, **kw)


def attn_bwd_vdim(q, k, v, o, lse, do, c, **kw):
    """Backward with v, o, do [B,H,n,v] of their own width (the same call as attn_bwd)."""
    return attn_bwd(q, k, v, o, lse, do, c, **kw)


def attn_fp8_quantize(q, k, v, signs=None, stream=None):
    """Block quantization to E4M3 for ``attn_fwd_fp8_blocks``: q, k, v bf16/fp16 [B,H,n,d]
    (d 64 or 128, n a multiple of 16); ``signs`` an int8 CUDA tensor of d entries turns on
    incoherent processing of q and k.  Returns (q8, k8, vt8, q_scales, k_scales, v_scales):
    E4M3 [B,H,n,d], [B,H,n,d], [B,H,d,n] and float32 [B,H,ceil(n/128)]."""
    B, H, n, d = _shape(q, k, v)
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q, k, v must be bfloat16 or float16")
    if signs is not None:
        if signs.dtype != torch.int8 or not signs.is_cuda or signs.numel() != d:
            raise ValueError("signs must be an int8 CUDA tensor of d entries")
        signs = signs.contiguous()
    f8 = getattr(torch, "float8_e4m3fn", torch.uint8)
    q8 = torch.empty((B, H, n, d), dtype=f8, device=q.device)
    k8 = torch.empty((B, H, n, d), dtype=f8, device=q.device)
    vt8 = torch.empty((B, H, d, n), dtype=f8, device=q.device)
    nb = (n + 127) // 128
    sq, sk, sv = (torch.empty((B, H, nb), dtype=torch.float32, device=q.device) for _ in range(3))
    _check(load().attn_fp8_quantize(DTYPE_CODE[q.dtype], B, H, n, d, _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(signs), _ptr(q8), _ptr(k8), _ptr(vt8), _ptr(sq),
                                    _ptr(sk), _ptr(sv), _stream_ptr(stream)))
    return q8, k8, vt8, sq, sk, sv


def attn_fwd_fp8_blocks(q8, k8, vt8, q_scales, k_scales, v_scales, c, mask="none",
                        mask_bits=None, mask_head_stride_words=0, o=None, lse=None, stream=None):
    """FP8 forward with one float32 scale per 128-row block of Q, K and V ([B,H,ceil(n/128)]
    CUDA tensors, as ``attn_fp8_quantize`` returns them); returns (o bfloat16 [B,H,n,d], lse)."""
    q8, k8, vt8 = (_fp8_bytes(t, nm) for t, nm in ((q8, "q8"), (k8, "k8"), (vt8, "vt8")))
    if q8.dim() != 4 or k8.shape != q8.shape:
        raise ValueError("q8 and k8 must be [B,H,n,d]")
    B, H, n, d = q8.shape
    if tuple(vt8.shape) != (B, H, d, n):
        raise ValueError("vt8 must be [B,H,d,n] (V transposed)")
    nb = (n + 127) // 128
    for t, nm in ((q_scales, "q_scales"), (k_scales, "k_scales"), (v_scales, "v_scales")):
        if (t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous()
                or tuple(t.shape) != (B, H, nb)):
            raise ValueError(f"{nm} must be a contiguous float32 CUDA tensor [B,H,ceil(n/128)]")
    kind, bits, row_words, hs = _mask_args(mask, mask_bits, mask_head_stride_words)
    if o is None:
        o = torch.empty((B, H, n, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, n), dtype=torch.float32, device=q8.device)
    _check(load().attn_fwd_fp8_blocks(B, H, n, d, float(c), _ptr(q8), _ptr(k8), _ptr(vt8),
                                      _ptr(q_scales), _ptr(k_scales), _ptr(v_scales), kind,
                                      _ptr(bits), row_words, hs, _ptr(o), _ptr(lse),
                                      _stream_ptr(stream)))
    return o, lse


def attn_merge(o_parts, lse_parts, dtype=torch.float32, o=None, lse=None, stream=None):
    """Merge partial results over disjoint key sets: o_parts [P, ..., d] float32 and
    lse_parts [P, ...] float32 -> (o [..., d] of ``dtype``, lse [...] float32)."""
    if o_parts.dtype != torch.float32 or lse_parts.dtype != torch.float32:
        raise ValueError("o_parts and lse_parts must be float32")
    if not (o_parts.is_cuda and o_parts.is_contiguous() and lse_parts.is_cuda
            and lse_parts.is_contiguous()):
        raise ValueError("o_parts and lse_parts must be contiguous CUDA tensors")
    if o_parts.shape[:-1] != lse_parts.shape:
        raise ValueError("o_parts must be lse_parts' shape plus a trailing d")
    parts, d = o_parts.shape[0], o_parts.shape[-1]
    rows = lse_parts[0].numel()
    if o is None:
        o = torch.empty(o_parts.shape[1:], dtype=dtype, device=o_parts.device)
    if lse is None:
        lse = torch.empty(lse_parts.shape[1:], dtype=torch.float32, device=o_parts.device)
    _check(load().attn_merge(DTYPE_CODE[o.dtype], parts, rows, d, _ptr(o_parts), _ptr(lse_parts),
                             _ptr(o), _ptr(lse), _stream_ptr(stream)))
    return o, lse


def attn_fwd_dropout(q, k, v, c, dropout_p, seed, **kw):
    """attn_fwd with dropout: the C entry point of the same name (see attn_fwd)."""
    if not dropout_p:
        raise ValueError("attn_fwd_dropout needs dropout_p > 0 (use attn_fwd otherwise)")
    return attn_fwd(q, k, v, c, dropout_p=dropout_p, seed=seed, **kw)


def attn_bwd_dropout(q, k, v, o, lse, do, c, dropout_p, seed, **kw):
    """attn_bwd replaying the dropout mask of attn_fwd_dropout for the same seed."""
    if not dropout_p:
        raise ValueError("attn_bwd_dropout needs dropout_p > 0 (use attn_bwd otherwise)")
    return attn_bwd(q, k, v, o, lse, do, c, dropout_p=dropout_p, seed=seed, **kw)


def attn_bwd_workspace_bytes(dtype, B, H, n, d) -> int:
    code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load().attn_bwd_workspace_bytes(code, B, H, n, d))


def attn_bwd(q, k, v, o, lse, do, c, mask="none", mask_bits=None, mask_head_stride_words=0,
             kv_block=0, dq=None, dk=None, dv=None, workspace=None, stream=None, dropout_p=0.0,
             seed=0):
    """Backward pass (vector-Jacobian product for upstream ``do``); returns (dq, dk, dv).
    dropout_p and seed must be those of the forward (attn_bwd_dropout replays its mask).
    v, o, do and dv may be narrower or wider than q and k (attn_bwd_vdim)."""
    B, H, n, d, v_dim = _shape_v(q, k, v)
    kind, bits, row_words, hs = _mask_args(mask, mask_bits, mask_head_stride_words)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = attn_bwd_workspace_bytes(q.dtype, B, H, n, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    lib = load()
    if v_dim != d:
        _check(lib.attn_bwd_vdim(DTYPE_CODE[q.dtype], B, H, n, d, v_dim, float(c), _ptr(q),
                                 _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), kind, _ptr(bits),
                                 row_words, hs, int(kv_block), float(dropout_p),
                                 int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(dq), _ptr(dk), _ptr(dv),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream_ptr(stream)))
        return dq, dk, dv
    if dropout_p:
        _check(lib.attn_bwd_dropout(DTYPE_CODE[q.dtype], B, H, n, d, float(c), _ptr(q), _ptr(k),
                                    _ptr(v), _ptr(o), _ptr(lse), _ptr(do), kind, _ptr(bits),
                                    row_words, hs, int(kv_block), float(dropout_p),
                                    int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(dq), _ptr(dk), _ptr(dv),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream_ptr(stream)))
        return dq, dk, dv
    _check(lib.attn_bwd(DTYPE_CODE[q.dtype], B, H, n, d, float(c), _ptr(q), _ptr(k), _ptr(v),
                        _ptr(o), _ptr(lse), _ptr(do), kind, _ptr(bits), row_words, hs,
                        int(kv_block), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                        workspace.numel() * workspace.element_size(), _stream_ptr(stream)))
    return dq, dk, dv


def attn_bwd_noalloc(q, k, v, o, lse, do, c, mask="none", mask_bits=None,
                     mask_head_stride_words=0, kv_block=0, dq=None, dk=None, dv=None, stream=None):
    """attn_bwd for callers that cannot allocate device memory when they run the backward.

    Same result as attn_bwd, but the float32 scratch comes from a fixed static array inside
    the library (ATTN_BWD_NOALLOC_SCRATCH_BYTES, 32 MiB), so no workspace is passed and the
    library allocates nothing.  Problems needing more scratch are refused with
    ATTN_ERR_WORKSPACE.  Calls that overlap on the GPU share that array and race; the first
    call on a device should come before any stream capture there.  Output tensors that are
    not given are allocated here with PyTorch, so a caller that must not allocate passes
    dq, dk and dv.
    """
    lib = load()
    if getattr(lib.attn_bwd_noalloc, "argtypes", None) is None:
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.attn_bwd_noalloc.argtypes = [i32, i32, i32, i32, i32, f32, vp, vp, vp, vp, vp, vp,
                                         i32, vp, i64, i64, i32, vp, vp, vp, vp]
        lib.attn_bwd_noalloc.restype = i32
    B, H, n, d = _shape(q, k, v)
    kind, bits, row_words, hs = _mask_args(mask, mask_bits, mask_head_stride_words)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(lib.attn_bwd_noalloc(DTYPE_CODE[q.dtype], B, H, n, d, float(c), _ptr(q), _ptr(k),
                                _ptr(v), _ptr(o), _ptr(lse), _ptr(do), kind, _ptr(bits),
                                row_words, hs, int(kv_block), _ptr(dq), _ptr(dk), _ptr(dv),
                                _stream_ptr(stream)))
    return dq, dk, dv


def attn_selftest_wait_timeout(stream=None) -> int:
    """Launch the library's failure-path self-test (a bounded wait that must time out)."""
    lib = load()
    lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_void_p]
    lib.attn_selftest_wait_timeout.restype = ctypes.c_int
    return _check(lib.attn_selftest_wait_timeout(_stream_ptr(stream)))


def attn_selftest_exp2(x, stream=None):
    """(2^x on the FMA pipe, 2^x on the MUFU unit) for a float32 CUDA tensor x (attn_selftest_exp2)."""
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    y_fma, y_mufu = torch.empty_like(x), torch.empty_like(x)
    _check(load().attn_selftest_exp2(_ptr(x), _ptr(y_fma), _ptr(y_mufu), x.numel(),
                                     _stream_ptr(stream)))
    return y_fma, y_mufu


def attn_debug_set_ring_stages(stages: int) -> None:
    """Cap every kernel's shared-memory ring depth at ``stages`` (0 = default); a testing aid:
    results are bit for bit the same at every depth (attn_debug_set_ring_stages)."""
    _check(load().attn_debug_set_ring_stages(int(stages)))


def attn_device_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device status word (see the header)."""
    return _check(load().attn_device_status(_stream_ptr(stream)))


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, c, mask, mask_bits, kv_block, dropout_p, seed):
        o, lse = attn_fwd(q, k, v, c, mask, mask_bits, 0, kv_block, dropout_p=dropout_p,
                          seed=seed)
        ctx.save_for_backward(q, k, v, o, lse, mask_bits)
        ctx.c, ctx.mask, ctx.kv_block, ctx.dropout_p, ctx.seed = c, mask, kv_block, dropout_p, seed
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse, mask_bits = ctx.saved_tensors
        dq, dk, dv = attn_bwd(q, k, v, o, lse, do.contiguous(), ctx.c, ctx.mask, mask_bits, 0,
                              ctx.kv_block, dropout_p=ctx.dropout_p, seed=ctx.seed)
        return dq, dk, dv, None, None, None, None, None, None


def attention(q, k, v, c, mask="none", mask_bits=None, kv_block=0, dropout_p=0.0, seed=0):
    """Differentiable exact attention O = softmax(c QKᵀ + mask) V, with optional dropout on
    the probabilities (the backward replays the forward's mask for ``seed``); v may have its
    own width (q, k [B,H,n,d], v [B,H,n,v])."""
    return _Attention.apply(q, k, v, c, mask, mask_bits, kv_block, dropout_p, seed)
