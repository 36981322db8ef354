"""Float64 CPU oracle for the batched temperature -> min-p -> top-k -> top-p -> sample chain.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline may import this package. The product (``nucleus_token_sampler_gb300``) never imports it
and shares no code with it.

The arithmetic lives in ``tps_oracle.c`` (plain C, float64, no fast-math, no FMA contraction);
this module only builds it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tps_oracle.c")
_LIB = os.path.join(_HERE, "libtps_oracle.so")
_lock = threading.Lock()
_default = None

ROW_OK, ROW_NAN, ROW_ALL_MASKED, ROW_BAD_PARAM = 0, 1, 2, 3
FLAG_TOPP_BAND, FLAG_MINP_BAND, FLAG_RACE_BAND = 1, 2, 4
FLAG_ACCEPT_BAND = 8                                  # speculative acceptance: u Q(x) within rounding of P(x)
FLAG_DRAFT_TOPP_BAND, FLAG_DRAFT_MINP_BAND = 16, 32   # the draft row's own band flags


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle (gcc, OpenMP, float64, -ffp-contract=off) into a shared library."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes view of one build of the oracle library (the default build, or a test's variant)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P = ctypes.c_void_p
        lib.tpso_sample.restype = ctypes.c_int
        lib.tpso_sample.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P, P, P, P, P,
                                    P, ctypes.c_uint64, P, P, P, P, P, P, P, ctypes.c_int]
        lib.tpso_sample_rejection.restype = ctypes.c_int
        lib.tpso_sample_rejection.argtypes = lib.tpso_sample.argtypes + [P]
        lib.tpso_uniform_round.restype = ctypes.c_double
        lib.tpso_uniform_round.argtypes = [ctypes.c_uint64] * 4 + [ctypes.c_uint32]
        lib.tpso_uniform.restype = ctypes.c_double
        lib.tpso_uniform.argtypes = [ctypes.c_uint64] * 4
        lib.tpso_uniform_spec.restype = ctypes.c_double
        lib.tpso_uniform_spec.argtypes = [ctypes.c_uint64] * 4
        lib.tpso_spec_accept.restype = ctypes.c_int
        lib.tpso_spec_accept.argtypes = [P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P, P, P, P, P, P, P, P,
                                         P, P, P, ctypes.c_uint64, P, P, P, P, P, P, ctypes.c_int]
        lib.tpso_philox4x32_10.restype = None
        lib.tpso_philox4x32_10.argtypes = [P, P, P]
        lib.tpso_max_threads.restype = ctypes.c_int
        I64 = ctypes.c_int64
        lib.tpso_penalties.restype = ctypes.c_int
        lib.tpso_penalties.argtypes = [P, ctypes.c_int, I64, I64, I64, P, I64, I64, P, P, P, P, P]
        self.lib = lib
        self.path = lib_path

    def sample(self, z, temperature, top_k, top_p, min_p, seed, step=0, *, row_ids=None,
               want_probs=False, nthreads=0, draw="race"):
        """Run the oracle on a [B, V] array of logits (widened exactly to float64).

        ``temperature``, ``top_p`` and ``min_p`` are rounded to float32 first (the values the GPU
        receives) and then widened, so both sides see the same numbers.  Returns a dict of numpy
        arrays: token, status, cutoff, kept, flags, z_s, z_k, n_s (+ probs when asked).

        ``draw="rejection"`` draws each row by sort-free rejection rounds instead of one race over
        the kept set (same kept set and distribution, other uniforms) and adds ``rounds``.
        """
        z = np.ascontiguousarray(np.asarray(z, dtype=np.float64))
        if z.ndim != 2:
            raise ValueError("z must be [B, V]")
        B, V = z.shape

        def vec(x, dt):
            return np.ascontiguousarray(np.broadcast_to(np.asarray(x), (B,)).astype(dt))

        T = vec(np.asarray(temperature, dtype=np.float32), np.float64)
        P = vec(np.asarray(top_p, dtype=np.float32), np.float64)
        M = vec(np.asarray(min_p, dtype=np.float32), np.float64)
        K = vec(top_k, np.int32)
        S = vec(np.asarray(seed).astype(np.uint64), np.uint64)
        R = None if row_ids is None else vec(row_ids, np.int64)
        out = {
            "token": np.empty(B, np.int32),
            "status": np.empty(B, np.int32),
            "cutoff": np.empty(B, np.float64),
            "kept": np.empty(B, np.int32),
            "flags": np.empty(B, np.int32),
        }
        aux = np.empty((B, 3), np.float64)
        probs = np.empty((B, V), np.float64) if want_probs else None
        args = (_ptr(z), B, V, V, _ptr(T), _ptr(K), _ptr(P), _ptr(M), _ptr(S), _ptr(R),
                int(step) & ((1 << 64) - 1), _ptr(out["token"]), _ptr(probs), _ptr(out["status"]),
                _ptr(out["cutoff"]), _ptr(out["kept"]), _ptr(out["flags"]), _ptr(aux), int(nthreads))
        if draw == "race":
            rc = self.lib.tpso_sample(*args)
        elif draw == "rejection":
            out["rounds"] = np.zeros(B, np.int32)
            rc = self.lib.tpso_sample_rejection(*args, _ptr(out["rounds"]))
        else:
            raise ValueError("draw must be 'race' or 'rejection'")
        if rc != 0:
            raise MemoryError("oracle scratch allocation failed")
        out["z_s"], out["z_k"], out["n_s"] = aux[:, 0].copy(), aux[:, 1].copy(), aux[:, 2].copy()
        if want_probs:
            out["probs"] = probs
        return out

    def spec_accept(self, zt, zd, target, draft, draft_token, seed, step=0, *, row_ids=None, nthreads=0):
        """Speculative acceptance of one draft token per row.

        ``zt``, ``zd``: [B, V] target and draft logits (widened exactly to float64); ``target`` and
        ``draft``: (temperature, top_k, top_p, min_p), each a scalar or [B] (T, p and min_p rounded to
        float32 first, as the GPU receives them); ``draft_token``: [B] the token the draft sampled.
        Returns token, accepted, status, flags, p_x (P of the draft token) and q_x (Q of it)."""
        zt = np.ascontiguousarray(np.asarray(zt, dtype=np.float64))
        zd = np.ascontiguousarray(np.asarray(zd, dtype=np.float64))
        if zt.ndim != 2 or zt.shape != zd.shape:
            raise ValueError("zt and zd must both be [B, V]")
        B, V = zt.shape

        def vec(x, dt):
            return np.ascontiguousarray(np.broadcast_to(np.asarray(x), (B,)).astype(dt))

        def params(t):
            T, k, p, m = t
            return (vec(np.asarray(T, dtype=np.float32), np.float64), vec(k, np.int32),
                    vec(np.asarray(p, dtype=np.float32), np.float64), vec(np.asarray(m, dtype=np.float32), np.float64))

        Tt, kt, pt, mt = params(target)
        Td, kd, pd, md = params(draft)
        X = vec(draft_token, np.int32)
        S = vec(np.asarray(seed).astype(np.uint64), np.uint64)
        R = None if row_ids is None else vec(row_ids, np.int64)
        out = {k: np.empty(B, np.int32) for k in ("token", "accepted", "status", "flags")}
        out["p_x"] = np.empty(B, np.float64)
        out["q_x"] = np.empty(B, np.float64)
        rc = self.lib.tpso_spec_accept(_ptr(zt), _ptr(zd), B, V, V, _ptr(Tt), _ptr(kt), _ptr(pt), _ptr(mt), _ptr(Td),
                                       _ptr(kd), _ptr(pd), _ptr(md), _ptr(X), _ptr(S), _ptr(R),
                                       int(step) & ((1 << 64) - 1), _ptr(out["token"]), _ptr(out["accepted"]),
                                       _ptr(out["status"]), _ptr(out["flags"]), _ptr(out["p_x"]), _ptr(out["q_x"]),
                                       int(nthreads))
        if rc != 0:
            raise MemoryError("oracle scratch allocation failed")
        return out

    def uniform_spec(self, seed: int, row: int, step: int, token: int) -> float:
        """The speculative acceptance's uniform for (seed, row, step, token); token 2^20 - 1 is the
        acceptance test's own."""
        m = (1 << 64) - 1
        return self.lib.tpso_uniform_spec(seed & m, row & m, step & m, token & m)

    def penalties(self, z, history, hist_len=None, repetition=None, frequency=None, presence=None,
                  bf16=False):
        """Repetition, frequency and presence penalties on raw logits (float32 arithmetic).

        ``z``: [B, V] logits as float32 values (bfloat16 logits widened exactly, with ``bf16`` set
        so results are rounded back to bfloat16); ``history``: [B, H] int32 token ids (entries
        outside [0, V) ignored); ``hist_len``: [B] or None (every row uses H); the three penalty
        vectors: [B] float32 or None (off).  Returns (penalised logits as float32, row status).
        """
        z = np.array(z, dtype=np.float32, order="C", copy=True)
        B, V = z.shape
        h = np.ascontiguousarray(np.asarray(history, dtype=np.int32).reshape(B, -1))
        H = h.shape[1]

        def vec(x, dt):
            return None if x is None else np.ascontiguousarray(np.broadcast_to(np.asarray(x, dtype=dt), (B,)))

        L, R, F, Pr = vec(hist_len, np.int32), vec(repetition, np.float32), vec(frequency, np.float32), \
            vec(presence, np.float32)
        st = np.empty(B, np.int32)
        rc = self.lib.tpso_penalties(_ptr(z), int(bool(bf16)), B, V, V, _ptr(h), H, H, _ptr(L), _ptr(R), _ptr(F),
                                     _ptr(Pr), _ptr(st))
        if rc != 0:
            raise MemoryError("oracle scratch allocation failed")
        return z, st

    def uniform(self, seed: int, row: int, step: int, token: int) -> float:
        """The race's uniform u in (0, 1) for (seed, row, step, token)."""
        m = (1 << 64) - 1
        return self.lib.tpso_uniform(seed & m, row & m, step & m, token & m)

    def uniform_round(self, seed: int, row: int, step: int, token: int, rnd: int) -> float:
        """The rejection draw's uniform for (seed, row, step, token) in round `rnd`."""
        m = (1 << 64) - 1
        return self.lib.tpso_uniform_round(seed & m, row & m, step & m, token & m, rnd)

    def philox4x32_10(self, counter, key):
        """One Philox4x32-10 block: counter = 4 x uint32, key = 2 x uint32 -> 4 x uint32."""
        c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint32))
        k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
        o = np.empty(4, np.uint32)
        self.lib.tpso_philox4x32_10(_ptr(c), _ptr(k), _ptr(o))
        return o

    def max_threads(self) -> int:
        return int(self.lib.tpso_max_threads())


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def sample(*args, **kwargs):
    return default().sample(*args, **kwargs)


def uniform(seed: int, row: int, step: int, token: int) -> float:
    return default().uniform(seed, row, step, token)


def penalties(*args, **kwargs):
    return default().penalties(*args, **kwargs)


def spec_accept(*args, **kwargs):
    return default().spec_accept(*args, **kwargs)


def philox4x32_10(counter, key):
    return default().philox4x32_10(counter, key)


def max_threads() -> int:
    return default().max_threads()
