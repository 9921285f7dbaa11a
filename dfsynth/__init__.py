"""Seeded synthetic inputs for the Dual-Flow decode step.

This module is the one piece shared by the GPU side (tests, bench) and the CPU
oracle side: it draws tensor elements from a counter-based hash (see synth.h)
and holds none of the method's arithmetic. Every element is a pure function of
(seed, tensor name, flat index), so a host fill of any slice reproduces the
exact bits a device fill wrote in place.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
HOST_LIB = os.path.join(_BUILD, "libdfsynth_host.so")
CUDA_LIB = os.path.join(_BUILD, "libdfsynth_cuda.so")

NVCC_ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def build(verbose: bool = False) -> None:
    """Compile the host (gcc + OpenMP) and device (nvcc, sm_103a) fill libraries in-tree."""
    os.makedirs(_BUILD, exist_ok=True)
    cmds = [
        ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11",
         os.path.join(_HERE, "synth_host.c"), "-o", HOST_LIB],
        ["nvcc", *NVCC_ARCH, "-O3", "-lineinfo", "-shared", "-Xcompiler", "-fPIC", "-fmad=false",
         os.path.join(_HERE, "synth_cuda.cu"), "-o", CUDA_LIB],
    ]
    for c in cmds:
        if verbose:
            print(" ".join(c))
        subprocess.run(c, check=True)


_host = None
_cuda = None


def _host_lib():
    global _host
    if _host is None:
        if not os.path.exists(HOST_LIB):
            build()
        lib = ctypes.CDLL(HOST_LIB)
        u64, f32, i32 = ctypes.c_uint64, ctypes.c_float, ctypes.c_int32
        vp = ctypes.c_void_p
        lib.dfs_fill_normal_bf16.argtypes = [vp, u64, u64, u64, u64, f32]
        lib.dfs_fill_normal_f32.argtypes = [vp, u64, u64, u64, u64, f32]
        lib.dfs_fill_uniform_i32.argtypes = [vp, u64, u64, u64, u64, i32, i32]
        lib.dfs_permutation_i32.argtypes = [vp, u64, u64, u64]
        for f in (lib.dfs_fill_normal_bf16, lib.dfs_fill_normal_f32, lib.dfs_fill_uniform_i32,
                  lib.dfs_permutation_i32):
            f.restype = None
        _host = lib
    return _host


def _cuda_lib():
    global _cuda
    if _cuda is None:
        if not os.path.exists(CUDA_LIB):
            raise RuntimeError(f"{CUDA_LIB} missing: run dfsynth.build()")
        lib = ctypes.CDLL(CUDA_LIB)
        u64, f32, vp = ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p
        for f in (lib.dfs_cuda_fill_normal_bf16, lib.dfs_cuda_fill_normal_f32):
            f.argtypes = [vp, u64, u64, u64, u64, f32, vp]
            f.restype = ctypes.c_int
        _cuda = lib
    return _cuda


def tensor_id(name: str) -> int:
    """FNV-1a 64-bit hash of the tensor's name: the per-tensor stream id."""
    h = 0xCBF29CE484222325
    for ch in name.encode():
        h ^= ch
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def _scale(sigma: float) -> float:
    return float(np.float32(sigma / 65536.0))


def host_normal(seed: int, name: str, shape, sigma: float, dtype: str, offset: int = 0) -> np.ndarray:
    """N(0, sigma^2) draws (Irwin-Hall) for elements [offset, offset + prod(shape)) of tensor `name`.

    dtype 'bf16' returns the raw bf16 bit patterns as uint16; 'f32' returns float32.
    """
    shape = tuple(int(s) for s in np.atleast_1d(shape))
    n = int(np.prod(shape)) if shape else 1
    lib = _host_lib()
    if dtype == "bf16":
        out = np.empty(n, dtype=np.uint16)
        lib.dfs_fill_normal_bf16(out.ctypes.data, seed, tensor_id(name), offset, n, _scale(sigma))
    elif dtype == "f32":
        out = np.empty(n, dtype=np.float32)
        lib.dfs_fill_normal_f32(out.ctypes.data, seed, tensor_id(name), offset, n, _scale(sigma))
    else:
        raise ValueError(dtype)
    return out.reshape(shape)


def host_gain(seed: int, name: str, shape, sigma: float, dtype: str) -> np.ndarray:
    """Norm gains: exactly 1.0 when sigma == 0, else 1 + N(0, sigma^2) rounded to the storage dtype."""
    shape = tuple(int(s) for s in np.atleast_1d(shape))
    if sigma == 0.0:
        g = np.ones(shape, dtype=np.float32)
    else:
        g = np.float32(1.0) + host_normal(seed, name, shape, sigma, "f32")
    return f32_to_bf16_bits(g) if dtype == "bf16" else g.astype(np.float32)


def host_uniform_int(seed: int, name: str, n: int, lo: int, hi: int, offset: int = 0) -> np.ndarray:
    """Integers uniform on [lo, hi] (inclusive), element i = lo + word(i) mod (hi - lo + 1)."""
    out = np.empty(int(n), dtype=np.int32)
    _host_lib().dfs_fill_uniform_i32(out.ctypes.data, seed, tensor_id(name), offset, int(n), lo, hi)
    return out


def host_permutation(seed: int, name: str, n: int) -> np.ndarray:
    """A seeded Fisher-Yates permutation of 0..n-1."""
    out = np.empty(int(n), dtype=np.int32)
    _host_lib().dfs_permutation_i32(out.ctypes.data, seed, tensor_id(name), int(n))
    return out


def cuda_normal_(ptr: int, seed: int, name: str, numel: int, sigma: float, dtype: str, offset: int = 0,
                 stream: int = 0) -> None:
    """Fill `numel` elements at device address `ptr` in place (same bits as host_normal)."""
    lib = _cuda_lib()
    fn = lib.dfs_cuda_fill_normal_bf16 if dtype == "bf16" else lib.dfs_cuda_fill_normal_f32
    rc = fn(ctypes.c_void_p(ptr), seed, tensor_id(name), offset, int(numel), _scale(sigma), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"dfsynth device fill failed: cuda error {rc}")


# ---- storage-format helpers (representation only) ----------------------------------------

def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)
