"""fp64 CPU oracle for paged attention over a block-tabled KV cache.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline / reference leg may import this package.  It
shares no code with the CUDA library: ``oracle.c`` is compiled on its own with
gcc and loaded here through ctypes; tensors are passed as raw host bytes.

What each function computes, and the page passage it follows, is written at
the top of ``oracle.c``:

* ``reshape_and_cache`` -- slot-mapping scatter (TensorSharp "Mistral 3" page,
  section 11: fresh K/V written to ``blockId * blockSize + offset``);
* ``copy_blocks`` -- whole-block copy used for prefix-cache reuse (mistral.rs
  page, paged-attention / prefix-cache section);
* ``paged_attention`` -- gather through the block table, then dense two-pass
  softmax attention in double (section 11's "gather, then flash attention",
  with the causal GQA attention of sections 3 and 4.1);
* ``dense_attention`` -- the same math on a contiguous per-sequence cache
  (section 10's [NumKVHeads, maxSeqLen, headDim] layout), used only to check
  the paged oracle's gather.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "oracle.c"
_LIB_PATH = _HERE / "_liboracle.so"

F32, F16, BF16 = 0, 1, 2

_lib = None


def build(force: bool = False) -> Path:
    """Compile oracle.c into oracle/_liboracle.so with gcc (OpenMP if present)."""
    if _LIB_PATH.exists() and not force and _LIB_PATH.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB_PATH
    tmp = _LIB_PATH.with_suffix(f".{os.getpid()}.tmp")
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", str(_SRC), "-o", str(tmp), "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(str(build()))
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.oracle_decode_elem.argtypes = [vp, i64, i32]
        lib.oracle_decode_elem.restype = ctypes.c_double
        lib.oracle_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32]
        lib.oracle_copy_blocks.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32]
        lib.oracle_paged_attention.argtypes = [vp, vp, i32, vp, i32, vp, vp, i32, vp, i32, vp,
                                               i32, i32, i32, i32, i32, f32]
        lib.oracle_dense_attention.argtypes = [vp, vp, i32, vp, i32, vp, vp, i32, vp, i32, i32,
                                               i32, f32]
        lib.oracle_num_threads.argtypes = []
        for name in ("oracle_reshape_and_cache", "oracle_copy_blocks", "oracle_paged_attention",
                     "oracle_dense_attention", "oracle_num_threads"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


_CODES = {"float32": F32, "torch.float32": F32, "float16": F16, "torch.float16": F16,
          "torch.bfloat16": BF16}


def _dtype_code(x) -> int:
    try:
        return _CODES[str(x.dtype)]
    except KeyError:
        raise TypeError(f"oracle: unsupported element type {x.dtype}") from None


def _host(x, writable: bool = False) -> np.ndarray:
    """A contiguous host ndarray over the same bytes (torch CPU tensor or ndarray)."""
    if isinstance(x, np.ndarray):
        arr = x
    else:  # torch tensor on the CPU: reinterpret 16-bit floats as raw int16
        if x.device.type != "cpu" or not x.is_contiguous():
            raise ValueError("oracle: inputs must be contiguous CPU tensors")
        t = x
        if t.element_size() == 2 and t.is_floating_point():
            import torch
            t = t.view(torch.int16)
        arr = t.numpy()
    if not arr.flags["C_CONTIGUOUS"]:
        raise ValueError("oracle: inputs must be C-contiguous")
    if writable and not arr.flags["WRITEABLE"]:
        raise ValueError("oracle: output buffer is read-only")
    return arr


def _ptr(arr: np.ndarray) -> int:
    return arr.ctypes.data


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: error {rc} (bad argument or index)")


def num_threads() -> int:
    """Threads the oracle's OpenMP region uses (1 when built without OpenMP)."""
    return int(_load().oracle_num_threads())


def decode_elements(raw: np.ndarray, dtype_code: int) -> np.ndarray:
    """Widen every element of ``raw`` (uint16 / float32 bytes) to double, one call each."""
    lib = _load()
    arr = np.ascontiguousarray(raw)
    return np.array([lib.oracle_decode_elem(_ptr(arr), i, dtype_code) for i in range(arr.size)])


def reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, block_size: int) -> None:
    """In place on host pools ``[NB][bs][Hkv][D]``: scatter ``key/value [T][Hkv][D]``."""
    k, v = _host(key), _host(value)
    kc, vc = _host(key_cache, True), _host(value_cache, True)
    sm = np.ascontiguousarray(_host(slot_mapping), dtype=np.int64)
    T, Hkv, D = key.shape
    NB = key_cache.shape[0]
    _check(_load().oracle_reshape_and_cache(_ptr(k), _ptr(v), _ptr(kc), _ptr(vc), _ptr(sm), T,
                                            Hkv, D, block_size, NB, _dtype_code(key_cache)),
           "reshape_and_cache")


def copy_blocks(key_cache, value_cache, block_mapping, block_size: int) -> None:
    """In place on host pools: copy whole blocks for each (src, dst) row of ``block_mapping``."""
    kc, vc = _host(key_cache, True), _host(value_cache, True)
    bm = np.ascontiguousarray(_host(block_mapping), dtype=np.int64)
    NB, bs, Hkv, D = key_cache.shape
    assert bs == block_size
    _check(_load().oracle_copy_blocks(_ptr(kc), _ptr(vc), _ptr(bm), bm.shape[0], Hkv, D,
                                      block_size, NB, _dtype_code(key_cache)), "copy_blocks")


def paged_attention(query, query_start_loc, key_cache, value_cache, block_tables, context_lens,
                    scale: float) -> np.ndarray:
    """Attention of packed query rows ``[Tq][Hq][D]`` over the paged cache; returns fp64.

    Decode is the case ``query_start_loc = [0, 1, ..., S]``.
    """
    q = _host(query)
    kc, vc = _host(key_cache), _host(value_cache)
    qsl = np.ascontiguousarray(_host(query_start_loc), dtype=np.int32)
    bt = np.ascontiguousarray(_host(block_tables), dtype=np.int32)
    cl = np.ascontiguousarray(_host(context_lens), dtype=np.int32)
    Tq, Hq, D = query.shape
    NB, bs, Hkv, _ = key_cache.shape
    S = cl.shape[0]
    out = np.zeros((Tq, Hq, D), dtype=np.float64)
    _check(_load().oracle_paged_attention(_ptr(out), _ptr(q), _dtype_code(query), _ptr(qsl), S,
                                          _ptr(kc), _ptr(vc), _dtype_code(key_cache), _ptr(bt),
                                          bt.shape[1] if bt.ndim == 2 else 0, _ptr(cl), Hq, Hkv,
                                          D, bs, NB, float(scale)), "paged_attention")
    return out


def dense_attention(query, query_start_loc, k_dense: np.ndarray, v_dense: np.ndarray,
                    context_lens, scale: float) -> np.ndarray:
    """Attention over contiguous fp64 caches ``[S][Hkv][Lmax][D]``; returns fp64."""
    q = _host(query)
    qsl = np.ascontiguousarray(_host(query_start_loc), dtype=np.int32)
    cl = np.ascontiguousarray(_host(context_lens), dtype=np.int32)
    kd = np.ascontiguousarray(k_dense, dtype=np.float64)
    vd = np.ascontiguousarray(v_dense, dtype=np.float64)
    Tq, Hq, D = query.shape
    S, Hkv, Lmax, _ = kd.shape
    out = np.zeros((Tq, Hq, D), dtype=np.float64)
    _check(_load().oracle_dense_attention(_ptr(out), _ptr(q), _dtype_code(query), _ptr(qsl), S,
                                          _ptr(kd), _ptr(vd), Lmax, _ptr(cl), Hq, Hkv, D,
                                          float(scale)), "dense_attention")
    return out
