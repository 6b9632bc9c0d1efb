"""Python binding of the paged KV-cache decode library (``_lib/libpkv.so``).

Argument marshalling only: every function checks tensor placement (all of a
call's CUDA tensors on one device, made current for the call), dtype, shape
and contiguity, then passes raw device pointers and that device's current
CUDA stream to the C ABI declared in ``include/pkv.h``.  All work runs in the
library's CUDA kernels; there is no CPU path.  A missing library raises.

    paged_kv_append(k, v, key_cache, value_cache, slot_mapping)
    paged_attention_decode(out, q, key_cache, value_cache, block_tables, seq_lens, scale, ...)
    copy_blocks(key_caches, value_caches, src_dst_pairs)
"""
from __future__ import annotations

import ctypes
import functools
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpkv.so")

PKV_OK, PKV_ERR_INVALID, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE, PKV_ERR_CUDA, PKV_ERR_OOM = range(6)
_DT = {torch.float16: 0, torch.bfloat16: 1}
_POOL_DT = {torch.float16: 0, torch.bfloat16: 1, torch.uint8: 2}   # uint8 pools hold E4M3 codes
PLAN_MAX_SEQS = 1024        # PKV_PLAN_MAX_SEQS: batches up to this size run through the plan kernel
PLANNED = 1                 # PKV_PLANNED: run over the plan an earlier call wrote
INPUTS_READY = 2            # PKV_INPUTS_READY: nothing pending writes the pools, tables, lengths or plan

# every symbol include/pkv.h declares
ABI_SYMBOLS = ("pkv_version", "pkv_last_error", "pkv_paged_kv_append", "pkv_decode_workspace_bytes",
               "pkv_decode_partition_tokens", "pkv_decode_plan_partition_tokens", "pkv_paged_attention_decode", "pkv_copy_blocks", "pkv_device_error",
               "pkv_paged_attention_decode_static", "pkv_swap_blocks", "pkv_paged_attention_verify", "pkv_bm_create", "pkv_bm_destroy",
               "pkv_bm_num_free_blocks", "pkv_bm_seq_len", "pkv_bm_refcount", "pkv_bm_allocate", "pkv_bm_fork",
               "pkv_bm_free", "pkv_bm_append_slots", "pkv_bm_block_tables", "pkv_paged_kv_append_fp8",
               "pkv_paged_attention_decode_fp8", "pkv_decode_plan", "pkv_paged_attention_decode_planned",
               "pkv_paged_attention_decode_fp8_planned", "pkv_paged_kv_append_decode",
               "pkv_paged_attention_verify_fp8")

_lib = None


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"pkv status {status}: {message}")
        self.status = status


def load() -> ctypes.CDLL:
    """Load the built library (build it with ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    c_i, c_i64, c_p, c_sz, c_f = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float
    lib.pkv_version.restype = c_i
    lib.pkv_version.argtypes = []
    lib.pkv_last_error.restype = ctypes.c_char_p
    lib.pkv_last_error.argtypes = []
    lib.pkv_paged_kv_append.restype = c_i
    lib.pkv_paged_kv_append.argtypes = [c_p, c_p, c_p, c_p, c_p, c_i64, c_i64, c_i, c_i, c_i, c_i, c_p]
    lib.pkv_decode_workspace_bytes.restype = c_sz
    lib.pkv_decode_workspace_bytes.argtypes = [c_i, c_i, c_i, c_i, c_i, c_i]
    lib.pkv_decode_partition_tokens.restype = c_i
    lib.pkv_decode_partition_tokens.argtypes = [c_i, c_i, c_i, c_i, c_i]
    lib.pkv_decode_plan_partition_tokens.restype = c_i
    lib.pkv_decode_plan_partition_tokens.argtypes = [c_p, c_i, c_i, c_i, c_p]
    lib.pkv_paged_attention_decode.restype = c_i
    lib.pkv_paged_attention_decode.argtypes = [c_p, c_p, c_p, c_p, c_p, c_i, c_p, c_i, c_i, c_i, c_i, c_i, c_i,
                                               c_i64, c_f, c_i, c_p, c_sz, c_i, c_p]
    lib.pkv_paged_attention_verify.restype = c_i
    lib.pkv_paged_attention_verify.argtypes = [c_p, c_p, c_p, c_p, c_p, c_i, c_p, c_i, c_i, c_i64, c_i, c_i, c_i,
                                               c_i, c_i64, c_f, c_i, c_i, c_p, c_sz, c_i, c_p]
    lib.pkv_paged_kv_append_fp8.restype = c_i
    lib.pkv_paged_kv_append_fp8.argtypes = [c_p, c_p, c_p, c_p, c_p, c_i64, c_i64, c_i, c_i, c_i, c_i, c_p, c_p, c_p]
    lib.pkv_paged_attention_decode_fp8.restype = c_i
    lib.pkv_paged_attention_decode_fp8.argtypes = [c_p, c_p, c_p, c_p, c_p, c_i, c_p, c_i, c_i, c_i, c_i, c_i, c_i,
                                                   c_i64, c_f, c_i, c_p, c_p, c_p, c_sz, c_i, c_p]
    lib.pkv_paged_attention_decode_fp8_planned.restype = c_i
    lib.pkv_paged_attention_decode_fp8_planned.argtypes = [c_p, c_p, c_p, c_p, c_p, c_i, c_p, c_i, c_i, c_i64, c_i,
                                                           c_i, c_i, c_i, c_i64, c_f, c_i, c_p, c_p, c_p, c_sz, c_i,
                                                           c_p]
    lib.pkv_paged_attention_decode_planned.restype = c_i
    lib.pkv_paged_attention_decode_planned.argtypes = [c_p, c_p, c_p, c_p, c_p, c_i, c_p, c_i, c_i, c_i64, c_i, c_i,
                                                       c_i, c_i, c_i64, c_f, c_i, c_p, c_sz, c_i, c_p]
    lib.pkv_paged_attention_verify_fp8.restype = c_i
    lib.pkv_paged_attention_verify_fp8.argtypes = [c_p, c_p, c_p, c_p, c_p, c_i, c_p, c_i, c_i, c_i64, c_i, c_i, c_i,
                                                   c_i, c_i64, c_f, c_i, c_p, c_p, c_i, c_p, c_sz, c_i, c_p]
    lib.pkv_paged_kv_append_decode.restype = c_i
    lib.pkv_paged_kv_append_decode.argtypes = [c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_i, c_p, c_i, c_i, c_i64, c_i,
                                               c_i, c_i, c_i, c_i64, c_f, c_i, c_i, c_p, c_p, c_p, c_sz, c_i, c_i, c_p]
    lib.pkv_decode_plan.restype = c_i
    lib.pkv_decode_plan.argtypes = [c_p, c_i, c_p, c_i, c_i, c_i64, c_i, c_i, c_i, c_i, c_i, c_p, c_sz, c_i, c_p]
    lib.pkv_copy_blocks.restype = c_i
    lib.pkv_copy_blocks.argtypes = [ctypes.POINTER(c_p), ctypes.POINTER(c_p), c_i, c_p, c_i64, c_i64, c_i, c_i,
                                    c_i, c_i, c_p]
    lib.pkv_device_error.restype = c_i
    lib.pkv_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint), c_i]
    lib.pkv_swap_blocks.restype = c_i
    lib.pkv_swap_blocks.argtypes = [ctypes.POINTER(c_p)] * 4 + [c_i, c_p, c_i64, c_i64, c_i64, c_i, c_i, c_i, c_i, c_p]
    lib.pkv_bm_create.restype = c_p
    lib.pkv_bm_create.argtypes = [c_i64, c_i, c_p]
    lib.pkv_bm_destroy.restype = None
    lib.pkv_bm_destroy.argtypes = [c_p]
    lib.pkv_bm_num_free_blocks.restype = c_i64
    lib.pkv_bm_num_free_blocks.argtypes = [c_p]
    lib.pkv_bm_seq_len.restype = c_i64
    lib.pkv_bm_seq_len.argtypes = [c_p, c_i64]
    lib.pkv_bm_refcount.restype = c_i
    lib.pkv_bm_refcount.argtypes = [c_p, c_i64]
    for name, args in (("pkv_bm_allocate", [c_p, c_i64, c_i64]), ("pkv_bm_fork", [c_p, c_i64, c_i64]),
                       ("pkv_bm_free", [c_p, c_i64]),
                       ("pkv_bm_append_slots", [c_p, c_p, c_i64, c_p, c_p, c_i64, c_p]),
                       ("pkv_bm_block_tables", [c_p, c_p, c_i64, c_p, c_i, ctypes.c_int32, c_p])):
        getattr(lib, name).restype = c_i
        getattr(lib, name).argtypes = args
    lib.pkv_paged_attention_decode_static.restype = c_i
    lib.pkv_paged_attention_decode_static.argtypes = [c_p, c_p, c_p, c_p, c_p, c_i, c_p, c_i, c_i, c_i, c_i, c_i, c_i,
                                                      c_i64, c_f, c_i, c_i, c_p]
    _lib = lib
    return lib


def _check(status: int):
    if status != PKV_OK:
        raise PkvError(status, load().pkv_last_error().decode(errors="replace"))


def _cuda_devices(values):
    """The CUDA devices of the tensors among ``values`` (tensors, or lists / tuples of them)."""
    devs = set()
    for v in values:
        for t in (v if isinstance(v, (list, tuple)) else (v,)):
            if isinstance(t, torch.Tensor) and t.is_cuda:
                devs.add(t.device)
    return devs


def _one_device(fn):
    """Every CUDA tensor of the call on one device, and that device current while
    the library runs: the kernels launch on the current device, on the stream of
    the tensors' device, and dereference every pointer there."""
    @functools.wraps(fn)
    def call(*args, **kwargs):
        devs = _cuda_devices(list(args) + list(kwargs.values()))
        if len(devs) > 1:
            raise ValueError(f"{fn.__name__}: tensors on more than one device: {sorted(str(d) for d in devs)}")
        if not devs:
            return fn(*args, **kwargs)
        with torch.cuda.device(devs.pop()):
            return fn(*args, **kwargs)
    return call


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _cuda(name, t, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


def _pool(name, c, dtypes=(torch.float16, torch.bfloat16)):
    _cuda(name, c, dtypes, 4)
    return c.shape  # num_blocks, block_size, num_kv_heads, head_dim


@_one_device
def paged_kv_append(k, v, key_cache, value_cache, slot_mapping) -> None:
    """Write k[t], v[t] ([T, Hkv, d]) into slot slot_mapping[t] (int64; < 0 = skip)."""
    NB, bs, Hkv, d = _pool("key_cache", key_cache)
    if value_cache.shape != key_cache.shape or value_cache.dtype != key_cache.dtype:
        raise ValueError("value_cache must match key_cache")
    args = [_cuda("k", k, key_cache.dtype, 3), _cuda("v", v, key_cache.dtype, 3), _cuda("key_cache", key_cache),
            _cuda("value_cache", value_cache), _cuda("slot_mapping", slot_mapping, torch.int64, 1)]
    T = k.shape[0]
    if tuple(k.shape) != (T, Hkv, d) or tuple(v.shape) != (T, Hkv, d) or slot_mapping.shape[0] != T:
        raise ValueError("k, v must be [T, num_kv_heads, head_dim] and slot_mapping [T]")
    _check(load().pkv_paged_kv_append(*args, T, NB, bs, Hkv, d, _DT[key_cache.dtype], _stream(key_cache)))


def decode_partition_tokens(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len) -> int:
    return int(load().pkv_decode_partition_tokens(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len))


@_one_device
def decode_plan_partition_tokens(workspace, num_seqs, num_heads, num_kv_heads) -> int:
    """Partition size the last decode call with ``workspace`` used (-1: unplanned batch); synchronises."""
    return int(load().pkv_decode_plan_partition_tokens(_cuda("workspace", workspace), num_seqs, num_heads,
                                                       num_kv_heads, _stream(workspace)))


def decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len, partition_tokens=0) -> int:
    n = load().pkv_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len, partition_tokens)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid decode shape")
    return int(n)


def alloc_workspace(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len, partition_tokens=0, device="cuda"):
    """A device buffer of the size the decode call needs."""
    n = decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len, partition_tokens)
    return torch.empty(n, dtype=torch.uint8, device=device)


@_one_device
def decode_plan(workspace, block_tables, seq_lens, num_heads, key_cache, max_seq_len, partition_tokens=0,
                sum_seq_lens=0) -> None:
    """The work list of a decode batch, once per step (``pkv_decode_plan``): the runs that pass
    ``planned=True`` over the same batch then skip the plan kernel.  ``key_cache`` gives the pool's
    shape and element type (uint8: E4M3).  ``sum_seq_lens``: the lengths' sum if known (sizes the
    grid tighter; the runs must pass the same value)."""
    NB, bs, Hkv, d = _pool("key_cache", key_cache, tuple(_POOL_DT))
    B = seq_lens.shape[0]
    _cuda("block_tables", block_tables, torch.int32, 2)
    _cuda("seq_lens", seq_lens, torch.int32, 1)
    _check(load().pkv_decode_plan(ctypes.c_void_p(block_tables.data_ptr()), block_tables.shape[1],
                                  ctypes.c_void_p(seq_lens.data_ptr()), B, int(max_seq_len), int(sum_seq_lens),
                                  num_heads, Hkv, d, bs,
                                  _POOL_DT[key_cache.dtype], _cuda("workspace", workspace),
                                  workspace.numel() * workspace.element_size(), int(partition_tokens),
                                  _stream(workspace)))


@_one_device
def paged_attention_decode(out, q, key_cache, value_cache, block_tables, seq_lens, scale=None, block_size=None,
                           num_kv_heads=None, max_seq_len=None, workspace=None, partition_tokens=0,
                           planned=False, sum_seq_lens=0) -> None:
    """out[s, h] = softmax(scale * q[s, h] . K) V over positions [0, seq_lens[s]) of KV head h // G.

    q, out: [B, Hq, d]; caches [NB, bs, Hkv, d]; block_tables int32 [B, W]; seq_lens int32 [B].
    ``max_seq_len`` is the host-known bound of seq_lens (read from the device
    if omitted, which synchronises).  ``workspace``: see ``alloc_workspace``
    (allocated here when omitted).  ``planned``: run over the work list
    ``decode_plan`` put in ``workspace`` for this batch (no plan kernel).
    """
    NB, bs, Hkv, d = _pool("key_cache", key_cache)
    if block_size is not None and block_size != bs:
        raise ValueError(f"block_size {block_size} != cache block size {bs}")
    if num_kv_heads is not None and num_kv_heads != Hkv:
        raise ValueError(f"num_kv_heads {num_kv_heads} != cache heads {Hkv}")
    if value_cache.shape != key_cache.shape or value_cache.dtype != key_cache.dtype:
        raise ValueError("value_cache must match key_cache")
    B, Hq, dq = q.shape
    if dq != d or tuple(out.shape) != (B, Hq, d):
        raise ValueError("q and out must be [B, num_heads, head_dim]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if max_seq_len is None:
        max_seq_len = int(seq_lens.max().item()) if B else 0
    ptrs = [_cuda("out", out, key_cache.dtype), _cuda("q", q, key_cache.dtype), _cuda("key_cache", key_cache),
            _cuda("value_cache", value_cache), _cuda("block_tables", block_tables, torch.int32, 2)]
    _cuda("seq_lens", seq_lens, torch.int32, 1)
    if block_tables.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_tables / seq_lens batch mismatch")
    if workspace is None:
        workspace = alloc_workspace(B, Hq, Hkv, d, int(max_seq_len), partition_tokens, q.device)
    ws_ptr = _cuda("workspace", workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    lens_arg = [ctypes.c_void_p(seq_lens.data_ptr()), B, int(max_seq_len)]
    if planned:
        _check(load().pkv_paged_attention_decode_planned(
            *ptrs, block_tables.shape[1], *lens_arg, int(sum_seq_lens), Hq, Hkv, d, bs, NB, float(scale),
            _DT[key_cache.dtype], ws_ptr, ws_bytes, int(partition_tokens), _stream(q)))
    else:
        _check(load().pkv_paged_attention_decode(
            *ptrs, block_tables.shape[1], *lens_arg, Hq, Hkv, d, bs, NB, float(scale), _DT[key_cache.dtype], ws_ptr,
            ws_bytes, int(partition_tokens), _stream(q)))


def _scales(name, t, Hkv):
    _cuda(name, t, torch.float32, 1)
    if t.shape[0] != Hkv:
        raise ValueError(f"{name} must have num_kv_heads = {Hkv} entries")
    return ctypes.c_void_p(t.data_ptr())


@_one_device
def paged_kv_append_fp8(k, v, key_cache, value_cache, slot_mapping, k_scale, v_scale) -> None:
    """Quantize k[t], v[t] ([T, Hkv, d], fp16 / bf16) into slot slot_mapping[t] of uint8 E4M3 pools:
    code = e4m3(float32(x) / scale[head]) (nearest even, saturating); k_scale, v_scale float32 [Hkv]."""
    NB, bs, Hkv, d = _pool("key_cache", key_cache, (torch.uint8,))
    if value_cache.shape != key_cache.shape or value_cache.dtype != torch.uint8:
        raise ValueError("value_cache must match key_cache")
    T = k.shape[0]
    if tuple(k.shape) != (T, Hkv, d) or v.shape != k.shape or v.dtype != k.dtype:
        raise ValueError("k and v must be [T, num_kv_heads, head_dim] of one dtype")
    args = [_cuda("k", k, (torch.float16, torch.bfloat16)), _cuda("v", v, k.dtype), _cuda("key_cache", key_cache),
            _cuda("value_cache", value_cache), _cuda("slot_mapping", slot_mapping, torch.int64, 1)]
    if slot_mapping.shape[0] != T:
        raise ValueError("slot_mapping must have T entries")
    _check(load().pkv_paged_kv_append_fp8(*args, T, NB, bs, Hkv, d, _DT[k.dtype], _scales("k_scale", k_scale, Hkv),
                                          _scales("v_scale", v_scale, Hkv), _stream(key_cache)))


@_one_device
def paged_attention_decode_fp8(out, q, key_cache, value_cache, block_tables, seq_lens, k_scale, v_scale, scale=None,
                               max_seq_len=None, workspace=None, partition_tokens=0, planned=False,
                               sum_seq_lens=0) -> None:
    """paged_attention_decode over uint8 E4M3 pools: K = e4m3(code) * k_scale[g], V = e4m3(code) * v_scale[g];
    q, out fp16 / bf16 [B, Hq, 128]; k_scale, v_scale float32 [Hkv]."""
    NB, bs, Hkv, d = _pool("key_cache", key_cache, (torch.uint8,))
    if value_cache.shape != key_cache.shape or value_cache.dtype != torch.uint8:
        raise ValueError("value_cache must match key_cache")
    B, Hq, dq = q.shape
    if dq != d or tuple(out.shape) != (B, Hq, d):
        raise ValueError("q and out must be [B, num_heads, head_dim]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if max_seq_len is None:
        max_seq_len = int(seq_lens.max().item()) if B else 0
    ptrs = [_cuda("out", out, (torch.float16, torch.bfloat16)), _cuda("q", q, out.dtype), _cuda("key_cache", key_cache),
            _cuda("value_cache", value_cache), _cuda("block_tables", block_tables, torch.int32, 2)]
    _cuda("seq_lens", seq_lens, torch.int32, 1)
    if block_tables.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_tables / seq_lens batch mismatch")
    if workspace is None:
        workspace = alloc_workspace(B, Hq, Hkv, d, int(max_seq_len), partition_tokens, q.device)
    ws_ptr = _cuda("workspace", workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    lens_arg = [ctypes.c_void_p(seq_lens.data_ptr()), B, int(max_seq_len)]
    rest = [Hq, Hkv, d, bs, NB, float(scale), _DT[q.dtype], _scales("k_scale", k_scale, Hkv),
            _scales("v_scale", v_scale, Hkv), ws_ptr, ws_bytes, int(partition_tokens), _stream(q)]
    if planned:
        _check(load().pkv_paged_attention_decode_fp8_planned(*ptrs, block_tables.shape[1], *lens_arg,
                                                             int(sum_seq_lens), *rest))
    else:
        _check(load().pkv_paged_attention_decode_fp8(*ptrs, block_tables.shape[1], *lens_arg, *rest))


@_one_device
def paged_kv_append_decode(out, q, k, v, key_cache, value_cache, slot_mapping, block_tables, seq_lens, scale=None,
                           max_seq_len=None, workspace=None, partition_tokens=0, planned=False, sum_seq_lens=0,
                           k_scale=None, v_scale=None, inputs_ready=False) -> None:
    """paged_kv_append of one new token per sequence (k, v [B, Hkv, d]; slot_mapping int64 [B], the slot of
    position seq_lens[s] - 1, or < 0 for none) then paged_attention_decode, in one launch.  uint8 pools hold
    E4M3 codes and take k_scale / v_scale as paged_kv_append_fp8 does.  ``inputs_ready`` (with ``planned``):
    the caller guarantees that no work still pending on the stream writes the pools, block tables, seq_lens or
    the workspace's plan (every layer of a step after the first), so the tile loads may start while the
    preceding kernel finishes (``PKV_INPUTS_READY``)."""
    if inputs_ready and not planned:
        raise ValueError("inputs_ready needs planned=True (a plan written by an earlier call)")
    kv8 = key_cache.dtype == torch.uint8
    NB, bs, Hkv, d = _pool("key_cache", key_cache, tuple(_POOL_DT))
    if value_cache.shape != key_cache.shape or value_cache.dtype != key_cache.dtype:
        raise ValueError("value_cache must match key_cache")
    B, Hq, dq = q.shape
    if dq != d or tuple(out.shape) != (B, Hq, d):
        raise ValueError("q and out must be [B, num_heads, head_dim]")
    if tuple(k.shape) != (B, Hkv, d) or tuple(v.shape) != (B, Hkv, d):
        raise ValueError("k and v must be [B, num_kv_heads, head_dim]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if max_seq_len is None:
        max_seq_len = int(seq_lens.max().item()) if B else 0
    qdt = (torch.float16, torch.bfloat16) if kv8 else key_cache.dtype
    ptrs = [_cuda("out", out, qdt), _cuda("q", q, out.dtype), _cuda("k", k, out.dtype, 3), _cuda("v", v, out.dtype, 3),
            _cuda("key_cache", key_cache), _cuda("value_cache", value_cache),
            _cuda("slot_mapping", slot_mapping, torch.int64, 1), _cuda("block_tables", block_tables, torch.int32, 2)]
    _cuda("seq_lens", seq_lens, torch.int32, 1)
    if block_tables.shape[0] != B or seq_lens.shape[0] != B or slot_mapping.shape[0] != B:
        raise ValueError("block_tables / seq_lens / slot_mapping batch mismatch")
    if kv8:
        scales = [_scales("k_scale", k_scale, Hkv), _scales("v_scale", v_scale, Hkv)]
    else:
        scales = [None, None]
    if workspace is None:
        workspace = alloc_workspace(B, Hq, Hkv, d, int(max_seq_len), partition_tokens, q.device)
    ws_ptr = _cuda("workspace", workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().pkv_paged_kv_append_decode(
        *ptrs, block_tables.shape[1], ctypes.c_void_p(seq_lens.data_ptr()), B, int(max_seq_len), int(sum_seq_lens),
        Hq, Hkv, d, bs, NB, float(scale), _DT[q.dtype], _POOL_DT[key_cache.dtype], *scales, ws_ptr, ws_bytes,
        int(partition_tokens), (PLANNED if planned else 0) | (INPUTS_READY if inputs_ready else 0), _stream(q)))


@_one_device
def paged_attention_verify(out, q, key_cache, value_cache, block_tables, seq_lens, scale=None, max_seq_len=None,
                           workspace=None, partition_tokens=0, sum_seq_lens=0, k_scale=None, v_scale=None) -> None:
    """Multi-query paged attention: q, out [B, nq, Hq, d]; query token i of sequence s attends over
    positions [0, seq_lens[s] - nq + i] (the last nq positions are the queries' own K/V).  uint8 pools
    hold E4M3 codes and take k_scale / v_scale (float32 [Hkv]) as paged_attention_decode_fp8 does."""
    kv8 = key_cache.dtype == torch.uint8
    NB, bs, Hkv, d = _pool("key_cache", key_cache, tuple(_POOL_DT))
    if value_cache.shape != key_cache.shape or value_cache.dtype != key_cache.dtype:
        raise ValueError("value_cache must match key_cache")
    if q.dim() != 4:
        raise ValueError("q must be [B, num_queries, num_heads, head_dim]")
    B, nq, Hq, dq = q.shape
    if dq != d or tuple(out.shape) != tuple(q.shape):
        raise ValueError("q and out must be [B, num_queries, num_heads, head_dim]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if max_seq_len is None:
        max_seq_len = int(seq_lens.max().item()) if B else 0
    qdt = (torch.float16, torch.bfloat16) if kv8 else key_cache.dtype
    ptrs = [_cuda("out", out, qdt), _cuda("q", q, out.dtype), _cuda("key_cache", key_cache),
            _cuda("value_cache", value_cache), _cuda("block_tables", block_tables, torch.int32, 2)]
    _cuda("seq_lens", seq_lens, torch.int32, 1)
    if block_tables.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_tables / seq_lens batch mismatch")
    if workspace is None:
        workspace = alloc_workspace(B, Hq * nq, Hkv, d, int(max_seq_len), partition_tokens, q.device)
    ws_ptr = _cuda("workspace", workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    lens_arg = [ctypes.c_void_p(seq_lens.data_ptr()), B, int(max_seq_len), int(sum_seq_lens)]
    if kv8:
        _check(load().pkv_paged_attention_verify_fp8(
            *ptrs, block_tables.shape[1], *lens_arg, Hq, Hkv, d, bs, NB, float(scale), _DT[q.dtype],
            _scales("k_scale", k_scale, Hkv), _scales("v_scale", v_scale, Hkv), nq, ws_ptr, ws_bytes,
            int(partition_tokens), _stream(q)))
    else:
        _check(load().pkv_paged_attention_verify(
            *ptrs, block_tables.shape[1], *lens_arg, Hq, Hkv, d, bs, NB, float(scale), _DT[key_cache.dtype], nq,
            ws_ptr, ws_bytes, int(partition_tokens), _stream(q)))


@_one_device
def copy_blocks(key_caches, value_caches, src_dst_pairs) -> None:
    """For each (src, dst) row of src_dst_pairs (int64 [Np, 2]): every layer's block dst = block src."""
    if isinstance(key_caches, torch.Tensor):
        key_caches, value_caches = [key_caches], [value_caches]
    if len(key_caches) != len(value_caches) or not key_caches:
        raise ValueError("need the same non-zero number of key and value caches")
    shape, dt = key_caches[0].shape, key_caches[0].dtype
    for i, (kc, vc) in enumerate(zip(key_caches, value_caches)):
        _pool(f"key_caches[{i}]", kc, tuple(_POOL_DT))
        _pool(f"value_caches[{i}]", vc, tuple(_POOL_DT))
        if kc.shape != shape or vc.shape != shape or kc.dtype != dt or vc.dtype != dt:
            raise ValueError("all caches must share shape and dtype")
    _cuda("src_dst_pairs", src_dst_pairs, torch.int64, 2)
    if src_dst_pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be [Np, 2]")
    n = len(key_caches)
    karr = (ctypes.c_void_p * n)(*[kc.data_ptr() for kc in key_caches])
    varr = (ctypes.c_void_p * n)(*[vc.data_ptr() for vc in value_caches])
    NB, bs, Hkv, d = shape
    _check(load().pkv_copy_blocks(karr, varr, n, ctypes.c_void_p(src_dst_pairs.data_ptr()), src_dst_pairs.shape[0],
                                  NB, bs, Hkv, d, _POOL_DT[dt], _stream(key_caches[0])))


def _addressable_pool(name, t):
    """A pool the GPU can address: a CUDA tensor or a pinned CPU tensor."""
    if not isinstance(t, torch.Tensor) or t.dim() != 4 or t.dtype not in _POOL_DT:
        raise ValueError(f"{name} must be a 4-D fp16 / bf16 / uint8 (E4M3) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    return t.data_ptr()


@_one_device
def swap_blocks(src_key_caches, src_value_caches, dst_key_caches, dst_value_caches, src_dst_pairs) -> None:
    """dst[dst_i] = src[src_i] for every (src_i, dst_i) row of src_dst_pairs (int64 [Np, 2], on the GPU),
    for every layer's K and V pool.  Pools are CUDA tensors or pinned host tensors (swap out / swap in)."""
    lists = [src_key_caches, src_value_caches, dst_key_caches, dst_value_caches]
    lists = [[x] if isinstance(x, torch.Tensor) else list(x) for x in lists]
    n = len(lists[0])
    if n == 0 or any(len(x) != n for x in lists):
        raise ValueError("need the same non-zero number of pools in every list")
    src_shape, dst_shape, dt = lists[0][0].shape, lists[2][0].shape, lists[0][0].dtype
    ptrs = []
    for li, (name, pools) in enumerate(zip(("src_key", "src_value", "dst_key", "dst_value"), lists)):
        want = src_shape if li < 2 else dst_shape
        for i, t in enumerate(pools):
            ptrs.append(_addressable_pool(f"{name}[{i}]", t))
            if t.shape != want or t.dtype != dt:
                raise ValueError("pools must share dtype; source pools one shape, destination pools another")
    if tuple(src_shape[1:]) != tuple(dst_shape[1:]):
        raise ValueError("source and destination blocks must have the same shape")
    _cuda("src_dst_pairs", src_dst_pairs, torch.int64, 2)
    if src_dst_pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be [Np, 2]")
    arrs = [(ctypes.c_void_p * n)(*ptrs[k * n:(k + 1) * n]) for k in range(4)]
    _, bs, Hkv, d = src_shape
    _check(load().pkv_swap_blocks(*arrs, n, ctypes.c_void_p(src_dst_pairs.data_ptr()), src_dst_pairs.shape[0],
                                  src_shape[0], dst_shape[0], bs, Hkv, d, _POOL_DT[dt], _stream(src_dst_pairs)))


class BlockManager:
    """The library's host block manager (``pkv_bm_*``): free list, reference
    counts, copy-on-write at a fork.  Host only; it produces the inputs of the
    decode step (tables, lengths, slots) and the copy pairs for copy_blocks."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        import numpy as np

        self._np = np
        self.block_size = int(block_size)
        self._order = None if free_order is None else np.ascontiguousarray(free_order, dtype=np.int64)
        ptr = None if self._order is None else self._order.ctypes.data
        self._h = load().pkv_bm_create(int(num_blocks), self.block_size, ptr)
        if not self._h:
            raise ValueError("bad block manager arguments")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            load().pkv_bm_destroy(h)
            self._h = None

    @property
    def num_free_blocks(self) -> int:
        return int(load().pkv_bm_num_free_blocks(self._h))

    def seq_len(self, seq_id) -> int:
        return int(load().pkv_bm_seq_len(self._h, int(seq_id)))

    def refcount(self, block) -> int:
        return int(load().pkv_bm_refcount(self._h, int(block)))

    def allocate(self, seq_id, num_tokens) -> None:
        _check(load().pkv_bm_allocate(self._h, int(seq_id), int(num_tokens)))

    def fork(self, parent_id, child_id) -> None:
        _check(load().pkv_bm_fork(self._h, int(parent_id), int(child_id)))

    def free(self, seq_id) -> None:
        _check(load().pkv_bm_free(self._h, int(seq_id)))

    def append_slots(self, seq_ids):
        """One new token per sequence: (slots int64 [n], cow_pairs int64 [k, 2])."""
        np = self._np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        slots = np.empty(len(ids), dtype=np.int64)
        cow = np.empty((max(1, len(ids)), 2), dtype=np.int64)
        n = ctypes.c_int64(0)
        _check(load().pkv_bm_append_slots(self._h, ids.ctypes.data, len(ids), slots.ctypes.data, cow.ctypes.data,
                                          cow.shape[0], ctypes.byref(n)))
        return slots, cow[:n.value].copy()

    def block_tables(self, seq_ids, max_blocks_per_seq, pad=-1):
        """(int32 [n, max_blocks_per_seq] tables padded with `pad`, int32 [n] lengths)."""
        np = self._np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        tables = np.empty((len(ids), max_blocks_per_seq), dtype=np.int32)
        lens = np.empty(len(ids), dtype=np.int32)
        _check(load().pkv_bm_block_tables(self._h, ids.ctypes.data, len(ids), tables.ctypes.data,
                                          int(max_blocks_per_seq), int(pad), lens.ctypes.data))
        return tables, lens


def device_error(reset: bool = True) -> int:
    """The device error word (synchronises the device): bit 0 out-of-range id skipped, bit 1 wait timeout."""
    v = ctypes.c_uint(0)
    _check(load().pkv_device_error(ctypes.byref(v), 1 if reset else 0))
    return int(v.value)
