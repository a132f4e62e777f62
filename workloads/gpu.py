"""Device-side copy of the synthetic key generator (``keygen.cu``).

Draws a workload's keys straight into device memory, bit-identical to
``Workload.head_keys`` on the host: the host builds the quantile and cos/sin
tables once and hands the same tables to the kernel.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "keygen.cu")
LIB_PATH = os.path.join(_HERE, "libkeygen.so")
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(_SRC) > os.path.getmtime(LIB_PATH):
        nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call([nvcc if os.path.exists(nvcc) else "nvcc", "-gencode",
                               "arch=compute_103a,code=sm_103a", "-O3", "-fmad=false", "-Xcompiler",
                               "-fPIC", "-shared", "-o", tmp, _SRC])
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        _lib.keygen_fill.restype = ctypes.c_int
        _lib.keygen_fill.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i64, i64, i64, i64, i64,
                                     i64, ctypes.c_uint64, i32, P]
    return _lib


_tables = {}


def _device_tables(wl, device):
    import torch
    import workloads
    key = (wl.rope_theta, wl.head_dim, wl.positions, wl.key_seed, str(device))
    if key not in _tables:
        C, S = wl.rope_tables()
        _tables.clear()
        _tables[key] = (torch.from_numpy(workloads.ninv_table()).to(device),
                        torch.from_numpy(np.ascontiguousarray(C)).to(device),
                        torch.from_numpy(np.ascontiguousarray(S)).to(device),
                        torch.from_numpy(wl.unit()).to(device))
    return _tables[key]


def fill(wl, out, p0: int, count: int, layout: str, stream=None):
    """Write keys of positions p0..p0+count-1 into a device fp16 tensor.

    layout "prefill": out is [B, L, H, count, D]; "decode": out is [count, B, L, H, D].
    """
    import torch
    B, L, H, D = wl.batch, wl.n_layers, wl.n_kv_heads, wl.head_dim
    if layout == "prefill":
        assert tuple(out.shape) == (B, L, H, count, D)
        sb, sl, sh, sp = L * H * count * D, H * count * D, count * D, D
    elif layout == "decode":
        assert tuple(out.shape) == (count, B, L, H, D)
        sb, sl, sh, sp = L * H * D, H * D, D, B * L * H * D
    else:
        raise ValueError(layout)
    assert out.dtype == torch.float16 and out.is_contiguous() and out.is_cuda
    ninv, C, S, unit = _device_tables(wl, out.device)
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = lib().keygen_fill(out.data_ptr(), ninv.data_ptr(), C.data_ptr(), S.data_ptr(),
                           unit.data_ptr(), B, L, H, D, p0, count, sb, sl, sh, sp, wl.key_seed,
                           int(wl.late_riser), s)
    if rc != 0:
        raise RuntimeError(f"keygen launch failed ({rc})")


def device_inputs(wl, device="cuda"):
    """(prefill [B,L,H,S,D] or None, decode [T,B,L,H,D]) fp16 tensors on the device."""
    import torch
    B, L, H, D = wl.batch, wl.n_layers, wl.n_kv_heads, wl.head_dim
    pre = None
    if wl.prefill > 0:
        pre = torch.empty((B, L, H, wl.prefill, D), dtype=torch.float16, device=device)
        fill(wl, pre, 0, wl.prefill, "prefill")
    dec = torch.empty((wl.decode, B, L, H, D), dtype=torch.float16, device=device)
    fill(wl, dec, wl.prefill, wl.decode, "decode")
    return pre, dec
