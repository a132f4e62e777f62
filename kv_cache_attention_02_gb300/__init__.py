"""GB300-native cumulative proxy-attention KV-cache eviction.

H2O-adapted, Keyformer-adapted (frozen Gumbel regulariser, annealed
temperature) and PyramidKV-adapted (per-layer budget taper) eviction as one
fused sm_103a decode step, plus tensor-core prompt scoring. This module is the
thin Python face of the C ABI in ``include/kvevict.h``: it only marshals
arguments (tensor pointers, sizes, the current CUDA stream) into
``libkvevict.so``. Every step of the method runs in the library's kernels;
there is no CPU or PyTorch fallback, and importing fails loudly when the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvevict.so")

OK, ERR_INVALID_ARG, ERR_BAD_STATE, ERR_CUDA, ERR_OOM, ERR_DEVICE_CHECK = 0, -1, -2, -3, -4, -5
SCORE_CUMULATIVE, SCORE_CURRENT = 0, 1
PREFILL_BULK, PREFILL_SEQUENTIAL = 0, 1
DECODE_AUTO, DECODE_STREAM, DECODE_RESIDENT = 0, 1, 2
MAX_LAYERS = 256
MAX_PREFILL = 16384

i32, i64, u64, f32, f64, P = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float,
                              ctypes.c_double, ctypes.c_void_p)


class Config(ctypes.Structure):
    """Mirror of ``kvevict_config``."""
    _fields_ = [("batch", i32), ("n_layers", i32), ("n_kv_heads", i32), ("head_dim", i32),
                ("avg_budget", i32), ("pyramid_beta", f64), ("layer_budgets", P), ("n_sink", i32),
                ("tau_init", f32), ("tau_end", f32), ("anneal_steps", i32), ("rope_theta", f64),
                ("seed", u64), ("max_prefill", i32), ("recent", i32), ("score_mode", i32),
                ("prefill_mode", i32), ("with_values", i32), ("decode_kernel", i32)]


class KVEvictError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"kvevict error {code}: {msg}")
        self.code = code


_lib = None

# every symbol the header declares, with its ctypes signature
SIGNATURES = {
    "kvevict_budgets": (ctypes.c_int, [i32, i32, i32, f64, P]),
    "kvevict_create": (ctypes.c_int, [P, P, P]),
    "kvevict_destroy": (ctypes.c_int, [P]),
    "kvevict_reset": (ctypes.c_int, [P, P]),
    "kvevict_test_stall_next_step": (ctypes.c_int, [P]),
    "kvevict_prefill": (ctypes.c_int, [P, P, i32, P]),
    "kvevict_prefill_ex": (ctypes.c_int, [P, P, i32, P, P]),
    "kvevict_prefill_kv": (ctypes.c_int, [P, P, P, i32, P, P]),
    "kvevict_step_kv": (ctypes.c_int, [P, P, P, P, P]),
    "kvevict_decode_kv": (ctypes.c_int, [P, P, P, i32, P, P]),
    "kvevict_read_values": (ctypes.c_int, [P, i32, i32, i32, P, P, P]),
    "kvevict_step": (ctypes.c_int, [P, P, P, P]),
    "kvevict_decode": (ctypes.c_int, [P, P, i32, P, P]),
    "kvevict_run_host": (ctypes.c_int, [P, P, i32, P, i32, P, P]),
    "kvevict_read_state": (ctypes.c_int, [P, i32, i32, i32, P, P, P, P, P, P]),
    "kvevict_check": (ctypes.c_int, [P, P]),
    "kvevict_flush": (ctypes.c_int, [P, P]),
    "kvevict_next_pos": (ctypes.c_int, [P, P]),
    "kvevict_layer_budget": (ctypes.c_int, [P, i32, P]),
    "kvevict_decode_kernel_for": (ctypes.c_int, [P, i32, P]),
    "kvevict_layer_stats": (ctypes.c_int, [P, i32, P, P, P, P]),
    "kvevict_device_bytes": (ctypes.c_int, [P, P]),
    "kvevict_state_bytes": (ctypes.c_int, [P, P]),
    "kvevict_save_state": (ctypes.c_int, [P, P, ctypes.c_size_t, P]),
    "kvevict_load_state": (ctypes.c_int, [P, P, ctypes.c_size_t, P]),
    "kvevict_last_error": (ctypes.c_char_p, []),
    "kvevict_prefill_scores_noalloc": (ctypes.c_int, [P, i32, i32, i32, P, P]),
}


def lib() -> ctypes.CDLL:
    """Load ``libkvevict.so`` (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                              "(python -c 'import __graft_entry__ as g; g.build()')")
        _lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(_lib, name)
            fn.restype = res
            fn.argtypes = args
    return _lib


def _check(rc: int):
    if rc != OK:
        raise KVEvictError(rc, lib().kvevict_last_error().decode())


def last_error() -> str:
    return lib().kvevict_last_error().decode()


def budgets(n_layers: int, avg_budget: int, n_sink: int, beta: float) -> list[int]:
    """Per-layer budget taper computed by the library (host only)."""
    out = (i32 * max(1, n_layers))()
    _check(lib().kvevict_budgets(n_layers, avg_budget, n_sink, beta, ctypes.addressof(out)))
    return list(out)[:n_layers]


def prefill_scores_noalloc(keys, colsum, stream=None):
    """Causal column sums of prompts with no device allocation.

    keys: device fp16 [heads, S, D]; colsum: device float32 [heads, S] (output).
    For callers that cannot allocate device memory; see the C declaration of
    kvevict_prefill_scores_noalloc for the size limit and sharing rules.
    """
    heads, S, D = (int(x) for x in keys.shape)
    assert tuple(colsum.shape) == (heads, S)
    _check(lib().kvevict_prefill_scores_noalloc(_ptr(keys), heads, S, D, _ptr(colsum),
                                                _stream(stream)))


def _ptr(t) -> int:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        assert t.flags["C_CONTIGUOUS"]
        return t.ctypes.data
    assert t.is_contiguous(), "tensor must be contiguous"
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


class KVEvict:
    """One handle: a device-resident eviction state for B x L x H cache rows."""

    def __init__(self, *, batch: int, n_layers: int, n_kv_heads: int, head_dim: int,
                 avg_budget: int = 512, pyramid_beta: float = 1.0, layer_budgets=None,
                 n_sink: int = 4, tau_init: float = 0.0, tau_end: float = 0.0,
                 anneal_steps: int = 0, rope_theta: float = 10000.0, seed: int = 0,
                 max_prefill: int = 0, recent: int = 0, score_mode: int = SCORE_CUMULATIVE,
                 prefill_mode: int = PREFILL_BULK, with_values: bool = False,
                 decode_kernel: int = DECODE_AUTO, stream=None):
        self._lb = None
        if layer_budgets is not None:
            self._lb = (i32 * n_layers)(*layer_budgets)
        self.cfg = Config(batch, n_layers, n_kv_heads, head_dim, avg_budget, pyramid_beta,
                          ctypes.addressof(self._lb) if self._lb is not None else None, n_sink,
                          tau_init, tau_end, anneal_steps, rope_theta, seed & (2 ** 64 - 1),
                          max_prefill, recent, score_mode, prefill_mode, int(bool(with_values)),
                          decode_kernel)
        self._h = P()
        _check(lib().kvevict_create(ctypes.addressof(self.cfg), _stream(stream),
                                    ctypes.addressof(self._h)))
        self.B, self.L, self.H, self.D = batch, n_layers, n_kv_heads, head_dim
        self.with_values = bool(with_values)
        self.budgets = [self.layer_budget(l) for l in range(n_layers)]

    # ------------------------------------------------------------------ lifecycle
    def close(self):
        if self._h:
            lib().kvevict_destroy(self._h)
            self._h = P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def reset(self, stream=None):
        _check(lib().kvevict_reset(self._h, _stream(stream)))

    # ------------------------------------------------------------------ the path
    def prefill(self, keys, evicted=None, stream=None, values=None):
        """keys (values): device fp16 [B, L, H, S, D]; evicted: device int32 [S, B, L, H] or None."""
        S = int(keys.shape[3]) if keys is not None else 0
        if self.with_values:
            _check(lib().kvevict_prefill_kv(self._h, _ptr(keys), _ptr(values), S, _ptr(evicted),
                                            _stream(stream)))
        else:
            _check(lib().kvevict_prefill_ex(self._h, _ptr(keys), S, _ptr(evicted), _stream(stream)))

    def step(self, k_new, evicted=None, stream=None, v_new=None):
        """k_new (v_new): device fp16 [B, L, H, D]; evicted: device int32 [B, L, H] or None."""
        if self.with_values:
            _check(lib().kvevict_step_kv(self._h, _ptr(k_new), _ptr(v_new), _ptr(evicted),
                                         _stream(stream)))
        else:
            _check(lib().kvevict_step(self._h, _ptr(k_new), _ptr(evicted), _stream(stream)))

    def decode(self, keys, evicted=None, stream=None, values=None):
        """keys (values): device fp16 [T, B, L, H, D]; evicted: device int32 [T, B, L, H] or None."""
        if self.with_values:
            _check(lib().kvevict_decode_kv(self._h, _ptr(keys), _ptr(values), int(keys.shape[0]),
                                           _ptr(evicted), _stream(stream)))
        else:
            _check(lib().kvevict_decode(self._h, _ptr(keys), int(keys.shape[0]), _ptr(evicted),
                                        _stream(stream)))

    def run_host(self, prefill_keys, decode_keys, evicted=None, stream=None):
        """End to end from host memory (pinned tensors or numpy uint16 arrays)."""
        S = int(prefill_keys.shape[3]) if prefill_keys is not None else 0
        T = int(decode_keys.shape[0]) if decode_keys is not None else 0
        _check(lib().kvevict_run_host(self._h, _ptr(prefill_keys), S, _ptr(decode_keys), T,
                                      _ptr(evicted), _stream(stream)))

    # ------------------------------------------------------------------ queries
    def read_state(self, b: int, l: int, h: int, stream=None):
        """(keys fp16-bits [n, D], scores f32 [n], gumbel f32 [n], positions i32 [n])."""
        cap = self.budgets[l] + 1 if 0 <= l < self.L else 1  # the library validates indices
        keys = np.zeros((cap, self.D), np.uint16)
        sc = np.zeros(cap, np.float32)
        g = np.zeros(cap, np.float32)
        pos = np.zeros(cap, np.int32)
        n = i32(0)
        _check(lib().kvevict_read_state(self._h, b, l, h, keys.ctypes.data, sc.ctypes.data,
                                        g.ctypes.data, pos.ctypes.data, ctypes.addressof(n),
                                        _stream(stream)))
        k = n.value
        return keys[:k], sc[:k], g[:k], pos[:k]

    def read_values(self, b: int, l: int, h: int, stream=None):
        """Value rows of one cache row, fp16 bits [n, D], in slot order."""
        cap = self.budgets[l] + 1 if 0 <= l < self.L else 1
        vals = np.zeros((cap, self.D), np.uint16)
        n = i32(0)
        _check(lib().kvevict_read_values(self._h, b, l, h, vals.ctypes.data, ctypes.addressof(n),
                                         _stream(stream)))
        return vals[: n.value]

    def flush(self, stream=None):
        """Apply the last step's pending compaction (one kernel launch)."""
        _check(lib().kvevict_flush(self._h, _stream(stream)))

    def test_stall_next_step(self):
        """Test hook: the next decode launch makes one bounded wait run out."""
        _check(lib().kvevict_test_stall_next_step(self._h))

    def check(self, stream=None):
        _check(lib().kvevict_check(self._h, _stream(stream)))

    @property
    def next_pos(self) -> int:
        p = i64(0)
        _check(lib().kvevict_next_pos(self._h, ctypes.addressof(p)))
        return p.value

    def decode_kernel_for(self, T: int) -> int:
        """DECODE_STREAM or DECODE_RESIDENT: the kernel a call of T steps runs."""
        k = i32(0)
        _check(lib().kvevict_decode_kernel_for(self._h, T, ctypes.addressof(k)))
        return k.value

    def layer_budget(self, l: int) -> int:
        b = i32(0)
        _check(lib().kvevict_layer_budget(self._h, l, ctypes.addressof(b)))
        return b.value

    def layer_stats(self, l: int) -> dict:
        """tokens_kept, stored_bytes, full_bytes and compression_ratio of layer l."""
        kept, stored, full, ratio = i32(0), ctypes.c_uint64(0), ctypes.c_uint64(0), ctypes.c_double(0)
        _check(lib().kvevict_layer_stats(self._h, l, ctypes.addressof(kept), ctypes.addressof(stored),
                                         ctypes.addressof(full), ctypes.addressof(ratio)))
        return {"tokens_kept": kept.value, "stored_bytes": stored.value, "full_bytes": full.value,
                "compression_ratio": ratio.value}

    def device_bytes(self) -> int:
        v = ctypes.c_size_t(0)
        _check(lib().kvevict_device_bytes(self._h, ctypes.addressof(v)))
        return v.value

    # ------------------------------------------------------- checkpoint / resume
    def state_bytes(self) -> int:
        v = ctypes.c_size_t(0)
        _check(lib().kvevict_state_bytes(self._h, ctypes.addressof(v)))
        return v.value

    def save_state(self, out=None, stream=None) -> np.ndarray:
        """Snapshot of the cache state as a uint8 host array (or into `out`)."""
        n = self.state_bytes()
        buf = np.empty(n, np.uint8) if out is None else out
        assert buf.dtype == np.uint8 and buf.flags["C_CONTIGUOUS"] and buf.size >= n
        _check(lib().kvevict_save_state(self._h, buf.ctypes.data, buf.size, _stream(stream)))
        return buf

    def load_state(self, snapshot, stream=None):
        """Replace the cache state with a snapshot from save_state."""
        buf = np.ascontiguousarray(snapshot, dtype=np.uint8)
        _check(lib().kvevict_load_state(self._h, buf.ctypes.data, buf.size, _stream(stream)))


def from_workload(wl, stream=None, with_values=False, decode_kernel=DECODE_AUTO) -> KVEvict:
    """Handle for a ``workloads.Workload`` configuration."""
    return KVEvict(batch=wl.batch, n_layers=wl.n_layers, n_kv_heads=wl.n_kv_heads,
                   head_dim=wl.head_dim, avg_budget=wl.avg_budget, pyramid_beta=wl.beta,
                   n_sink=wl.n_sink, tau_init=wl.tau_init, tau_end=wl.tau_end,
                   anneal_steps=wl.anneal_steps, rope_theta=wl.rope_theta, seed=wl.gumbel_seed,
                   max_prefill=wl.prefill, recent=getattr(wl, "recent", 0),
                   score_mode=getattr(wl, "score_mode", SCORE_CUMULATIVE),
                   prefill_mode=getattr(wl, "prefill_mode", PREFILL_BULK),
                   with_values=with_values, decode_kernel=decode_kernel, stream=stream)
