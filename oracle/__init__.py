"""Python access to the fp64 CPU oracle (``kvevict_oracle.c``).

TEST INFRASTRUCTURE. The oracle checks the CUDA library; only the test suite,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import it.
It shares no code with the CUDA path and never consumes anything the CUDA path
produced. This module only marshals numpy arrays into the C functions; every
step of the method runs in the C file, which cites the pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvevict_oracle.c")
_HDR = os.path.join(_HERE, "kvevict_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")

GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, OpenMP)."""
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *GCC_FLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None

P = ctypes.c_void_p
i32, i64, u64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double


class HeadCfg(ctypes.Structure):
    _fields_ = [("D", i32), ("budget", i32), ("n_sink", i32), ("layer", i32), ("head", i32),
                ("tau_init", f64), ("tau_end", f64), ("anneal_steps", i64),
                ("theta", f64), ("seed", u64), ("recent", i32), ("mode", i32),
                ("prefill_mode", i32)]


def use_library(path: str | None):
    """Point this module at another build of the oracle (None: the default).

    Used by the mutation tests, which compile copies of the oracle with a
    planted mistake and check that the pins catch it. Returns the previous
    library handle.
    """
    global _lib
    prev = _lib
    _lib = None
    if path is not None:
        _bind(ctypes.CDLL(path))
    return prev


def _restore(handle):
    global _lib
    _lib = handle


def lib():
    if _lib is None:
        # KVEVICT_ORACLE_LIB: a separately built oracle (the mutation tests use it)
        _bind(ctypes.CDLL(os.environ.get("KVEVICT_ORACLE_LIB") or build()))
    return _lib


def _bind(handle):
    global _lib
    _lib = handle
    sig = {
        "orc_budgets": (ctypes.c_int, [i32, i32, i32, f64, P]),
        "orc_splitmix64": (u64, [u64]),
        "orc_gumbel_hash": (u64, [u64, i64, i64, i64]),
        "orc_gumbel_of_hash": (ctypes.c_float, [u64]),
        "orc_gumbel": (ctypes.c_float, [u64, i64, i64, i64]),
        "orc_gumbel_many": (None, [u64, i64, i64, i64, i64, P]),
        "orc_tau": (f64, [f64, f64, i64, i64]),
        "orc_f32_to_f16": (ctypes.c_uint16, [ctypes.c_float]),
        "orc_f16_to_f64": (f64, [ctypes.c_uint16]),
        "orc_f32_to_f16_array": (None, [i64, P, P]),
        "orc_f16_to_f64_array": (None, [i64, P, P]),
        "orc_rope_consts": (None, [f64, i32, i64, P, P]),
        "orc_rotate_row": (None, [i32, P, P, P]),
        "orc_step_accumulate": (i32, [i32, i32, P, P, P, P, P, i64, ctypes.c_float, i32]),
        "orc_regularised": (None, [i32, P, P, f64, P]),
        "orc_argmin": (i32, [i32, P, i32, i32]),
        "orc_evict": (i32, [i32, i32, P, P, P, P, i32, f64]),
        "orc_values_append": (None, [i32, i32, P, P]),
        "orc_values_evict": (i32, [i32, i32, P, i32]),
        "orc_values_prefill_apply": (i32, [i32, i32, P, P, P]),
        "orc_prefill_colsum": (None, [i32, i32, P, P]),
        "orc_prefill_select": (i32, [i32, i32, i32, i32, P, P]),
        "orc_prefill_lastrow": (None, [i32, i32, P, P]),
        "orc_prefill_apply": (i32, [i32, i32, P, P, P, P, f64, P, P, P, P]),
        "orc_run_head": (i32, [P, i32, P, i32, P, P, P, P, P, P]),
        "orc_run_heads": (i32, [i32, P, i32, P, i32, P, P, i32, P, P, P, P, P, i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(_lib, name)
        fn.restype = res
        fn.argtypes = args


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# --------------------------------------------------------------------------- scalar helpers
def budgets(n_layers: int, avg_budget: int, n_sink: int, beta: float) -> list[int]:
    out = np.zeros(max(n_layers, 1), dtype=np.int32)
    rc = lib().orc_budgets(n_layers, avg_budget, n_sink, beta, _p(out))
    if rc != 0:
        raise ValueError("invalid pyramid budget parameters")
    return [int(v) for v in out[:n_layers]]


def splitmix64(x: int) -> int:
    return int(lib().orc_splitmix64(x & (2**64 - 1)))


def gumbel_hash(seed: int, layer: int, head: int, pos: int) -> int:
    return int(lib().orc_gumbel_hash(seed, layer, head, pos))


def gumbel_of_hash(h: int) -> float:
    """The frozen Gumbel value a 64-bit hash maps to (float32, as a Python float)."""
    return float(lib().orc_gumbel_of_hash(h & (2**64 - 1)))


def gumbel(seed: int, layer: int, head: int, p0: int, count: int = 1) -> np.ndarray:
    out = np.zeros(count, dtype=np.float32)
    lib().orc_gumbel_many(seed, layer, head, p0, count, _p(out))
    return out


def tau(tau_init: float, tau_end: float, anneal_steps: int, pos: int) -> float:
    return float(lib().orc_tau(tau_init, tau_end, anneal_steps, pos))


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.zeros(x.shape, dtype=np.uint16)
    lib().orc_f32_to_f16_array(x.size, _p(x), _p(out))
    return out


def f16_bits_to_f64(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.zeros(h.shape, dtype=np.float64)
    lib().orc_f16_to_f64_array(h.size, _p(h), _p(out))
    return out


def rope_consts(theta: float, D: int, delta: int) -> tuple[np.ndarray, np.ndarray]:
    c = np.zeros(D // 2, dtype=np.float32)
    s = np.zeros(D // 2, dtype=np.float32)
    lib().orc_rope_consts(theta, D, delta, _p(c), _p(s))
    return c, s


def rotate_row(row: np.ndarray, c: np.ndarray, s: np.ndarray) -> np.ndarray:
    r = np.ascontiguousarray(row, dtype=np.uint16).copy()
    lib().orc_rotate_row(r.size, _p(r), _p(np.ascontiguousarray(c, np.float32)),
                         _p(np.ascontiguousarray(s, np.float32)))
    return r


SCORE_CUMULATIVE, SCORE_CURRENT = 0, 1


def prefill_lastrow(keys: np.ndarray) -> np.ndarray:
    keys = np.ascontiguousarray(keys, dtype=np.uint16)
    S, D = keys.shape
    out = np.zeros(S, dtype=np.float64)
    lib().orc_prefill_lastrow(S, D, _p(keys), _p(out))
    return out


def prefill_colsum(keys: np.ndarray) -> np.ndarray:
    keys = np.ascontiguousarray(keys, dtype=np.uint16)
    S, D = keys.shape
    out = np.zeros(S, dtype=np.float64)
    lib().orc_prefill_colsum(S, D, _p(keys), _p(out))
    return out


# --------------------------------------------------------------------------- per-head state
@dataclass
class HeadParams:
    D: int
    budget: int
    n_sink: int
    layer: int
    head: int
    tau_init: float
    tau_end: float
    anneal_steps: int
    theta: float
    seed: int
    recent: int = 0
    mode: int = SCORE_CUMULATIVE
    prefill_mode: int = 0     # 0 bulk, 1 one step per prompt token

    def cstruct(self) -> HeadCfg:
        return HeadCfg(self.D, self.budget, self.n_sink, self.layer, self.head, self.tau_init,
                       self.tau_end, self.anneal_steps, self.theta, self.seed, self.recent,
                       self.mode, self.prefill_mode)


class OracleHead:
    """One head's state as numpy arrays, stepped by the C oracle.

    The decision of which slot to evict is a separate call (``evict``), so a
    test can check the oracle's own choice (``select``) before applying one.
    """

    def __init__(self, prm: HeadParams, extra_rows: int = 0, values: bool = False):
        self.prm = prm
        cap = prm.budget + 1 + extra_rows
        self.K = np.zeros((cap, prm.D), dtype=np.uint16)
        # value rows (keyformer page, KeyformerState.values), or None: keys only
        self.V = np.zeros((cap, prm.D), dtype=np.uint16) if values else None
        self.score = np.zeros(cap, dtype=np.float64)
        self.g = np.zeros(cap, dtype=np.float32)
        self.pos = np.zeros(cap, dtype=np.int32)
        self.r = np.zeros(cap, dtype=np.float64)
        self.n = 0
        self.next_pos = 0

    # prefill ---------------------------------------------------------------
    def prefill_scores(self, keys: np.ndarray):
        """Column sums, Gumbel values and regularised scores of a prompt."""
        S = keys.shape[0]
        colsum = prefill_lastrow(keys) if self.prm.mode == SCORE_CURRENT else prefill_colsum(keys)
        g = gumbel(self.prm.seed, self.prm.layer, self.prm.head, 0, S)
        t = tau(self.prm.tau_init, self.prm.tau_end, self.prm.anneal_steps, S - 1)
        r = colsum + t * g.astype(np.float64)
        return colsum, g, r

    def prefill_select(self, r: np.ndarray) -> np.ndarray:
        S = r.shape[0]
        mask = np.zeros(S, dtype=np.uint8)
        rc = lib().orc_prefill_select(S, self.prm.budget, self.prm.n_sink, self.prm.recent,
                                      _p(np.ascontiguousarray(r, np.float64)), _p(mask))
        if rc < 0:
            raise ValueError("not enough evictable rows")
        return mask

    def prefill_apply(self, keys, colsum, g, mask, values=None):
        keys = np.ascontiguousarray(keys, dtype=np.uint16)
        S = keys.shape[0]
        kept = S - int(mask.sum())
        if kept > self.K.shape[0]:
            raise ValueError("prefill keeps more rows than the state holds")
        mask = np.ascontiguousarray(mask, np.uint8)
        self.n = lib().orc_prefill_apply(S, self.prm.D, _p(keys),
                                         _p(np.ascontiguousarray(colsum, np.float64)),
                                         _p(np.ascontiguousarray(g, np.float32)),
                                         _p(mask), self.prm.theta,
                                         _p(self.K), _p(self.score), _p(self.g), _p(self.pos))
        if self.V is not None:
            vals = np.ascontiguousarray(values, dtype=np.uint16)
            assert vals.shape == keys.shape
            lib().orc_values_prefill_apply(S, self.prm.D, _p(vals), _p(mask), _p(self.V))
        self.next_pos = S

    def prefill(self, keys: np.ndarray, values: np.ndarray | None = None) -> np.ndarray:
        if self.prm.prefill_mode == 1:     # one step per prompt token
            return np.array([self.step(k, None if values is None else values[t])
                             for t, k in enumerate(keys)], dtype=np.int32)
        colsum, g, r = self.prefill_scores(keys)
        mask = self.prefill_select(r)
        self.prefill_apply(keys, colsum, g, mask, values)
        return mask

    # decode ----------------------------------------------------------------
    def accumulate(self, k_new: np.ndarray, v_new: np.ndarray | None = None) -> int:
        p = self.next_pos
        gn = float(gumbel(self.prm.seed, self.prm.layer, self.prm.head, p, 1)[0])
        k = np.ascontiguousarray(k_new, dtype=np.uint16)
        if self.V is not None:
            v = np.ascontiguousarray(v_new, dtype=np.uint16)
            assert v.shape == k.shape
            lib().orc_values_append(self.prm.D, self.n, _p(self.V), _p(v))
        self.n = lib().orc_step_accumulate(self.prm.D, self.n, _p(self.K), _p(self.score),
                                           _p(self.g), _p(self.pos), _p(k), p, gn, self.prm.mode)
        self.next_pos = p + 1
        return self.n

    def over_budget(self) -> bool:
        return self.n > self.prm.budget

    def regularised(self) -> np.ndarray:
        t = tau(self.prm.tau_init, self.prm.tau_end, self.prm.anneal_steps, self.next_pos - 1)
        lib().orc_regularised(self.n, _p(self.score), _p(self.g), t, _p(self.r))
        return self.r[: self.n].copy()

    def select(self) -> int:
        self.regularised()
        return int(lib().orc_argmin(self.n, _p(self.r), self.prm.n_sink, self.prm.recent))

    def evict(self, e: int):
        if not (self.prm.n_sink <= e < self.n - self.prm.recent):
            raise ValueError(f"slot {e} is not evictable")
        if self.V is not None:
            lib().orc_values_evict(self.prm.D, self.n, _p(self.V), e)
        self.n = lib().orc_evict(self.prm.D, self.n, _p(self.K), _p(self.score), _p(self.g),
                                 _p(self.pos), e, self.prm.theta)

    def step(self, k_new: np.ndarray, v_new: np.ndarray | None = None) -> int:
        """Append, accumulate and, when over budget, evict the oracle's own pick."""
        self.accumulate(k_new, v_new)
        if self.over_budget():
            e = self.select()
            self.evict(e)
            return e
        return -1

    def state(self):
        n = self.n
        return (self.K[:n].copy(), self.score[:n].copy(), self.g[:n].copy(), self.pos[:n].copy())

    def values(self) -> np.ndarray:
        """The kept value rows [n, D] in slot order (a value-carrying head only)."""
        return self.V[: self.n].copy()


def run_heads(params: list[HeadParams], prefill_keys: np.ndarray, decode_keys: np.ndarray,
              n_threads: int = 0):
    """Whole pass (prefill + decode) for many heads in parallel, own decisions.

    prefill_keys [nh, S, D] uint16, decode_keys [nh, T, D] uint16.
    Returns (evicted [nh, T], n [nh], K, score, g, pos, threads_used).
    """
    nh = len(params)
    D = params[0].D
    S = prefill_keys.shape[1] if prefill_keys is not None else 0
    T = decode_keys.shape[1]
    cap = max(p.budget for p in params) + 1
    cfgs = (HeadCfg * nh)(*[p.cstruct() for p in params])
    pk = np.ascontiguousarray(prefill_keys if S else np.zeros((nh, 0, D), np.uint16), np.uint16)
    dk = np.ascontiguousarray(decode_keys, np.uint16)
    ev = np.zeros((nh, T), dtype=np.int32)
    K = np.zeros((nh, cap, D), dtype=np.uint16)
    sc = np.zeros((nh, cap), dtype=np.float64)
    g = np.zeros((nh, cap), dtype=np.float32)
    pos = np.zeros((nh, cap), dtype=np.int32)
    n = np.zeros(nh, dtype=np.int32)
    used = lib().orc_run_heads(nh, ctypes.addressof(cfgs), S, _p(pk), T, _p(dk), _p(ev), cap,
                               _p(K), _p(sc), _p(g), _p(pos), _p(n), n_threads)
    return ev, n, K, sc, g, pos, int(used)
