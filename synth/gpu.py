"""GPU twin of the seeded generators (synth_gpu.cu): same counters, same bits.

Input generation only.  Built into synth/libsynth_gpu.so by ``build()``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_gpu.cu")
_LIB = os.path.join(_HERE, "libsynth_gpu.so")
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call([nvcc if os.path.exists(nvcc) else "nvcc", "-gencode", "arch=compute_103a,code=sm_103a",
                               "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, i32, u32, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_uint64
        lib.synth_normal_rows.argtypes = [vp, u64, u32, i32, vp, i32, i32, i32, i32, vp]
        lib.synth_normal_rows.restype = ctypes.c_int
        lib.synth_q_rows.argtypes = [vp, u64, u32, i32, i32, i32, i32, vp]
        lib.synth_q_rows.restype = ctypes.c_int
        _lib = lib
    return _lib


def _stream():
    return torch.cuda.current_stream().cuda_stream


def normal_rows(out: torch.Tensor, seed: int, stream: int, b0: int, pos: torch.Tensor | None = None,
                p_const: int = 0) -> torch.Tensor:
    """Fill fp32 out[i][j][d] with the normal at (stream, b0+i, (pos[i] or p_const)+j, d)."""
    assert out.is_cuda and out.dtype == torch.float32 and out.is_contiguous() and out.dim() == 3
    batch, n, dim = out.shape
    rc = _load().synth_normal_rows(out.data_ptr(), seed, stream, b0, pos.data_ptr() if pos is not None else None,
                                   p_const, batch, n, dim, _stream())
    if rc != 0:
        raise RuntimeError(f"synth_normal_rows: CUDA error {rc}")
    return out


def q_rows(out: torch.Tensor, seed: int, stream: int, b0: int) -> torch.Tensor:
    """Fill bf16 out[i][r][d] with bf16(normal(stream, b0+i, r, d))."""
    assert out.is_cuda and out.dtype == torch.bfloat16 and out.is_contiguous() and out.dim() == 3
    batch, rows, dim = out.shape
    rc = _load().synth_q_rows(out.data_ptr(), seed, stream, b0, batch, rows, dim, _stream())
    if rc != 0:
        raise RuntimeError(f"synth_q_rows: CUDA error {rc}")
    return out
