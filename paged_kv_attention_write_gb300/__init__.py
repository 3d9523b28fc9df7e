"""GB300 (sm_103a) paged attention over a block-tabled KV cache.

A thin ctypes binding over the C ABI in ``include/pa.h`` (``libpa.so``, built
in-tree by ``paged_kv_attention_write_gb300/build.py``).  The Python functions
carry the C names and do argument marshalling only: shapes come from the
tensors, pointers from ``data_ptr()``, the stream from torch's current CUDA
stream.  Every step of the computation runs in the CUDA kernels; there is no
CPU fallback.  If the library is missing, importing this package fails.

Operations (see ``include/pa.h`` for layouts, ownership and error behaviour):

* ``pa_reshape_and_cache`` -- write fresh K/V to their cache slots;
* ``pa_decode`` -- one query token per sequence, split-K + log-sum-exp reduce;
* ``pa_prefill_chunk`` -- chunked prefill, causal in the chunk, full over the prefix;
* ``pa_copy_blocks`` -- whole-block copies for prefix-cache reuse;
* ``pa_reshape_and_cache_rope`` / ``pa_decode_rope`` -- the same with rotary position
  embedding (GPT-J pairs, YaRN table from ``pa_rope_yarn_freqs``) fused into the key write
  and the decode query load.
"""
from __future__ import annotations

import ctypes
from pathlib import Path
from typing import Optional

import torch

__all__ = [
    "PAError", "pa_reshape_and_cache", "pa_decode_workspace_size", "pa_decode", "pa_decode_noalloc",
    "pa_prefill_chunk", "pa_copy_blocks", "pa_status_string", "pa_version", "library_path",
    "Rope", "pa_rope_yarn_freqs", "pa_reshape_and_cache_rope", "pa_decode_rope", "pa_decode_write",
    "PA_F32", "PA_F16", "PA_BF16",
]

PA_F32, PA_F16, PA_BF16 = 0, 1, 2
_DTYPES = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16}

_LIB_PATH = Path(__file__).resolve().parent / "libpa.so"
if not _LIB_PATH.exists():
    raise ImportError(
        f"{_LIB_PATH} is missing: build the CUDA library first "
        "(python paged_kv_attention_write_gb300/build.py); there is no fallback")
_lib = ctypes.CDLL(str(_LIB_PATH))

_vp, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_lib.pa_reshape_and_cache.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                      _vp, _vp]
_lib.pa_decode_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32]
_lib.pa_decode_workspace_size.restype = _sz
_lib.pa_decode.argtypes = [_vp, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                           _i32, _i32, _f32, _i32, _vp, _sz, _vp, _vp]
_lib.pa_decode_noalloc.argtypes = [_vp, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                   _i32, _i32, _i32, _f32, _i32, _vp, _vp]
_lib.pa_prefill_chunk.argtypes = [_vp, _i32, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _i32, _vp, _i32,
                                  _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32, _vp, _vp]
_lib.pa_copy_blocks.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp]
_lib.pa_decode_write.argtypes = [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32,
                                 _i32, _i32, _i32, _i32, _f32, _i32, _vp, _sz, _vp, _vp]
_lib.pa_status_string.argtypes = [_i32]
_lib.pa_status_string.restype = ctypes.c_char_p
_lib.pa_version.argtypes = []


class _PaRope(ctypes.Structure):
    _fields_ = [("freqs", _vp), ("rope_dim", _i32), ("q_scale_beta", _f32), ("q_scale_orig_ctx", _i32)]


_lib.pa_rope_yarn_freqs.argtypes = [_vp, _i32, _f32, _f32, _i32, _f32, _f32]
_lib.pa_reshape_and_cache_rope.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                           ctypes.POINTER(_PaRope), _vp, _vp]
_lib.pa_decode_rope.argtypes = [_vp, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                                _i32, _i32, _f32, _i32, ctypes.POINTER(_PaRope), _vp, _sz, _vp, _vp]
for _name in ("pa_reshape_and_cache", "pa_decode", "pa_decode_noalloc", "pa_prefill_chunk",
              "pa_copy_blocks", "pa_version", "pa_rope_yarn_freqs", "pa_reshape_and_cache_rope",
              "pa_decode_rope", "pa_decode_write"):
    getattr(_lib, _name).restype = _i32


class PAError(RuntimeError):
    """A PA_ERR_* code returned by the C ABI."""

    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {pa_status_string(code)} ({code})")
        self.code = code


def library_path() -> Path:
    return _LIB_PATH


def pa_status_string(code: int) -> str:
    return _lib.pa_status_string(int(code)).decode()


def pa_version() -> int:
    return int(_lib.pa_version())


def _check(code: int, what: str) -> None:
    if code != 0:
        raise PAError(code, what)


def _dt(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def pa_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, *, status=None,
                         stream=None) -> None:
    """key/value ``[T][Hkv][D]`` -> pools ``[NB][bs][Hkv][D]`` at ``slot_mapping`` (int64)."""
    T, Hkv, D = key.shape
    NB, bs = key_cache.shape[:2]
    _check(_lib.pa_reshape_and_cache(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                                     _ptr(slot_mapping), T, Hkv, D, bs, NB, _dt(key_cache),
                                     _ptr(status), _stream(stream)), "pa_reshape_and_cache")


def pa_decode_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                             max_context_len: int) -> int:
    return int(_lib.pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                             max_context_len))


def pa_decode(out, query, key_cache, value_cache, block_tables, context_lens, max_context_len: int,
              scale: float, *, workspace=None, status=None, stream=None) -> None:
    """out ``[S][Hq][D]`` = attention of query ``[S][Hq][D]`` over each sequence's cache."""
    S, Hq, D = query.shape
    NB, bs, Hkv, _ = key_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.pa_decode(_ptr(out), _dt(out), _ptr(query), _ptr(key_cache), _ptr(value_cache),
                          _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                          int(max_context_len), S, Hq, Hkv, D, bs, NB, float(scale),
                          _dt(key_cache), _ptr(workspace), ws_bytes, _ptr(status),
                          _stream(stream)), "pa_decode")


def pa_decode_write(out, query, key, value, slot_mapping, key_cache, value_cache, block_tables,
                    context_lens, max_context_len: int, scale: float, *, workspace=None, status=None,
                    stream=None) -> None:
    """pa_reshape_and_cache of each sequence's new token (key / value ``[S][Hkv][D]`` to
    ``slot_mapping[s]``) and pa_decode, in one launch."""
    S, Hq, D = query.shape
    NB, bs, Hkv, _ = key_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.pa_decode_write(_ptr(out), _dt(out), _ptr(query), _ptr(key), _ptr(value), _ptr(slot_mapping),
                                _ptr(key_cache), _ptr(value_cache), _ptr(block_tables), block_tables.shape[1],
                                _ptr(context_lens), int(max_context_len), S, Hq, Hkv, D, bs, NB, float(scale),
                                _dt(key_cache), _ptr(workspace), ws_bytes, _ptr(status), _stream(stream)),
           "pa_decode_write")


def pa_decode_noalloc(out, query, key_cache, value_cache, block_tables, context_lens,
                      max_context_len: int, scale: float, *, status=None, stream=None) -> None:
    """pa_decode with the library's static scratch instead of a caller workspace, for
    callers that cannot allocate device memory.  Calls that overlap on the GPU race."""
    S, Hq, D = query.shape
    NB, bs, Hkv, _ = key_cache.shape
    _check(_lib.pa_decode_noalloc(_ptr(out), _dt(out), _ptr(query), _ptr(key_cache),
                                  _ptr(value_cache), _ptr(block_tables), block_tables.shape[1],
                                  _ptr(context_lens), int(max_context_len), S, Hq, Hkv, D, bs, NB,
                                  float(scale), _dt(key_cache), _ptr(status), _stream(stream)),
           "pa_decode_noalloc")


def pa_prefill_chunk(out, query, query_start_loc, max_query_len: int, key_cache, value_cache,
                     block_tables, context_lens, max_context_len: int, scale: float, *,
                     status=None, stream=None) -> None:
    """out ``[Tq][Hq][D]``: chunk rows attend their prefix and, causally, their chunk."""
    Tq, Hq, D = query.shape
    NB, bs, Hkv, _ = key_cache.shape
    S = context_lens.shape[0]
    _check(_lib.pa_prefill_chunk(_ptr(out), _dt(out), _ptr(query), _ptr(query_start_loc), Tq,
                                 int(max_query_len), _ptr(key_cache), _ptr(value_cache),
                                 _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                                 int(max_context_len), S, Hq, Hkv, D, bs, NB, float(scale),
                                 _dt(key_cache), _ptr(status), _stream(stream)),
           "pa_prefill_chunk")


def pa_copy_blocks(key_cache, value_cache, block_mapping, *, status=None, stream=None) -> None:
    """Copy whole blocks (K and V) for each (src, dst) row of ``block_mapping`` (int64 [N][2])."""
    NB, bs, Hkv, D = key_cache.shape
    _check(_lib.pa_copy_blocks(_ptr(key_cache), _ptr(value_cache), _ptr(block_mapping),
                               block_mapping.shape[0], Hkv, D, bs, NB, _dt(key_cache),
                               _ptr(status), _stream(stream)), "pa_copy_blocks")


# ----------------------------------------------------------------------------- rotary embedding

def pa_rope_yarn_freqs(rope_dim: int, base: float, yarn_scale: float = 1.0, orig_ctx: int = 0,
                       beta_fast: float = 32.0, beta_slow: float = 1.0):
    """The RoPE frequency table (host, fp32 ``[rope_dim / 2]``), YaRN-corrected when
    ``yarn_scale != 1`` and ``orig_ctx > 0`` (``include/pa.h`` states the formula)."""
    import numpy as np
    out = np.empty(rope_dim // 2, dtype=np.float32)
    _check(_lib.pa_rope_yarn_freqs(out.ctypes.data, rope_dim, float(base), float(yarn_scale), int(orig_ctx),
                                   float(beta_fast), float(beta_slow)), "pa_rope_yarn_freqs")
    return out


class Rope:
    """Rotary-embedding arguments: ``freqs`` a device fp32 tensor ``[rope_dim / 2]``, the
    rotated width, and the position-dependent query scale (off when ``q_scale_orig_ctx`` is 0)."""

    def __init__(self, freqs: torch.Tensor, rope_dim: int, q_scale_beta: float = 0.0, q_scale_orig_ctx: int = 0):
        self.freqs, self.rope_dim = freqs, rope_dim
        self.q_scale_beta, self.q_scale_orig_ctx = q_scale_beta, q_scale_orig_ctx

    def _c(self):
        return _PaRope(self.freqs.data_ptr(), int(self.rope_dim), float(self.q_scale_beta), int(self.q_scale_orig_ctx))


def pa_reshape_and_cache_rope(key, value, key_cache, value_cache, slot_mapping, positions, rope: Rope, *,
                              status=None, stream=None) -> None:
    """pa_reshape_and_cache with each key row rotated at ``positions`` (int32 [T])."""
    T, Hkv, D = key.shape
    NB, bs = key_cache.shape[:2]
    r = rope._c()
    _check(_lib.pa_reshape_and_cache_rope(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                                          _ptr(slot_mapping), _ptr(positions), T, Hkv, D, bs, NB,
                                          _dt(key_cache), ctypes.byref(r), _ptr(status), _stream(stream)),
           "pa_reshape_and_cache_rope")


def pa_decode_rope(out, query, key_cache, value_cache, block_tables, context_lens, max_context_len: int,
                   scale: float, rope: Rope, *, workspace=None, status=None, stream=None) -> None:
    """pa_decode with the (unrotated) query rotated and scaled at position context_len - 1."""
    S, Hq, D = query.shape
    NB, bs, Hkv, _ = key_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    r = rope._c()
    _check(_lib.pa_decode_rope(_ptr(out), _dt(out), _ptr(query), _ptr(key_cache), _ptr(value_cache),
                               _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                               int(max_context_len), S, Hq, Hkv, D, bs, NB, float(scale), _dt(key_cache),
                               ctypes.byref(r), _ptr(workspace), ws_bytes, _ptr(status), _stream(stream)),
           "pa_decode_rope")
