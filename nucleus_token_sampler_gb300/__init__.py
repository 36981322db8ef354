"""GB300 batched token sampler: temperature -> min-p -> top-k -> top-p -> one token per row.

A thin Python view of the C ABI in ``include/tps.h`` (``libtps.so``, built in-tree for sm_103a).
This module only marshals torch tensors into pointers and the current CUDA stream; every step of
the sampler runs in the CUDA kernels. There is no CPU fallback: if the library is missing or was
built for another machine, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

__all__ = ["build", "load", "sample", "sample_rejection", "apply_penalties", "spec_accept", "TPS_F32", "TPS_BF16", "ROW_STATUS", "library_path", "max_vocab",
           "cluster_size", "kernels_per_call", "version"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_CSRC = os.path.join(_HERE, "csrc")
_LIB = os.path.join(_HERE, "libtps.so")
_INCLUDE = os.path.join(os.path.dirname(_HERE), "include")
# The ABI and launch code, and one translation unit per (kernel, element type): compiled in parallel.
_SOURCES = ["tps_api.cu", "tps_k_cluster_f32.cu", "tps_k_cluster_bf16.cu", "tps_k_stream_f32.cu",
            "tps_k_stream_bf16.cu", "tps_k_penalty.cu", "tps_k_spec.cu", "tps_k_reject.cu"]
_HEADERS = ["tps_device.cuh", "tps_common.cuh", "tps_cluster.cuh", "tps_stream.cuh", "tps_penalty.cuh",
            "tps_spec.cuh", "tps_reject.cuh", "tps_kernels.h"]
_NVCC = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
         "-Xcompiler", "-fPIC"]

TPS_F32, TPS_BF16 = 0, 1
ROW_STATUS = {0: "ok", 1: "nan", 2: "all_masked", 3: "bad_param", 4: "timeout"}
_ERRORS = {1: "invalid argument", 2: "unknown dtype", 3: "vocabulary too large", 4: "misaligned pointer",
           5: "CUDA runtime error", 6: "more scratch than the fixed array of tps_sample_noalloc holds"}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB


def _stale() -> bool:
    if not os.path.exists(_LIB):
        return True
    t = os.path.getmtime(_LIB)
    deps = [os.path.join(_CSRC, f) for f in _SOURCES + _HEADERS] + [os.path.join(_INCLUDE, "tps.h")]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile ``libtps.so`` for sm_103a with nvcc: the translation units in parallel, then one link."""
    if not force and not _stale():
        return _LIB
    objdir = os.path.join(_HERE, "_build", f"obj{os.getpid()}")
    os.makedirs(objdir, exist_ok=True)
    objs, procs = [], []
    for f in _SOURCES:
        o = os.path.join(objdir, f.replace(".cu", ".o"))
        cmd = _NVCC + (["-Xptxas=-v"] if verbose else []) + ["-c", "-o", o, os.path.join(_CSRC, f)]
        procs.append((f, subprocess.Popen(cmd)))
        objs.append(o)
    failed = [f for f, p in procs if p.wait() != 0]
    if failed:
        raise RuntimeError(f"nvcc failed on {', '.join(failed)}")
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(_NVCC + ["-shared", "-o", tmp] + objs, check=True)
    os.replace(tmp, _LIB)
    for o in objs:
        os.remove(o)
    os.rmdir(objdir)
    return _LIB


def load():
    """Load the CUDA library (building it first if it is missing or older than its sources)."""
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P, I64, I32, U64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64
            lib.tps_sample.restype = I32
            lib.tps_sample.argtypes = [P, I32, I64, I64, P, P, P, P, P, U64, P, P, P]
            lib.tps_sample_ex.restype = I32
            lib.tps_sample_ex.argtypes = [P, I32, I64, I64, I64, P, P, P, P, P, U64, P, P, P, P, P, P]
            lib.tps_sample_kernel.restype = I32
            lib.tps_sample_kernel.argtypes = [P, I32, I64, I64, I64, P, P, P, P, P, U64, P, P, P, P, P, I32, P]
            lib.tps_apply_penalties.restype = I32
            lib.tps_apply_penalties.argtypes = [P, I32, I64, I64, I64, P, I64, I64, P, P, P, P, P, P]
            lib.tps_sample_full.restype = I32
            lib.tps_sample_full.argtypes = [P, I32, I64, I64, I64, P, P, P, P, P, U64, P, P, P, P, P, P, I32, P, P,
                                            I32, P]
            lib.tps_sample_noalloc.restype = I32
            lib.tps_sample_noalloc.argtypes = lib.tps_sample_full.argtypes
            lib.tps_sample_stall_test.restype = I32
            lib.tps_sample_stall_test.argtypes = [P, I32, I64, I64, P, P, P, P, P, U64, P, P, I64, U64, P]
            lib.tps_sample_rejection.restype = I32
            lib.tps_sample_rejection.argtypes = [P, I32, I64, I64, I64, P, P, P, P, P, U64, P, P, P, P, P, P]
            lib.tps_spec_accept.restype = I32
            lib.tps_spec_accept.argtypes = [P, P, I32, I64, I64, I64, P, P, P, P, P, P, P, P, P, P, U64, P, P, P, P]
            lib.tps_max_vocab.restype = I64
            lib.tps_max_vocab.argtypes = [I32]
            lib.tps_cluster_size.restype = I32
            lib.tps_cluster_size.argtypes = [I32, I64, I64]
            lib.tps_kernels_per_call.restype = I32
            lib.tps_kernels_per_call.argtypes = [I32, I64, I64, I32]
            lib.tps_status_string.restype = ctypes.c_char_p
            lib.tps_status_string.argtypes = [I32]
            lib.tps_last_cuda_error.restype = I32
            lib.tps_last_cuda_error.argtypes = []
            lib.tps_version.restype = I32
            lib.tps_version.argtypes = []
            _lib = lib
    return _lib


def version() -> int:
    return int(load().tps_version())


def max_vocab(dtype: torch.dtype = torch.float32) -> int:
    return int(load().tps_max_vocab(_dtype_code(dtype)))


def cluster_size(dtype: torch.dtype, B: int, V: int) -> int:
    return int(load().tps_cluster_size(_dtype_code(dtype), B, V))


def kernels_per_call(dtype: torch.dtype, B: int, V: int, kernel: str = "auto") -> int:
    """Kernels one call launches for this shape and kernel choice (1, or 2 for a split batch)."""
    return int(load().tps_kernels_per_call(_dtype_code(dtype), B, V, KERNELS[kernel]))


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return TPS_F32
    if dt == torch.bfloat16:
        return TPS_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {dt}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(rc: int):
    if rc != 0:
        lib = load()
        extra = f" (cudaError {lib.tps_last_cuda_error()})" if rc == 5 else ""
        raise RuntimeError(f"tps_sample failed: {_ERRORS.get(rc, rc)}{extra}")


def _param(x, B, dtype, device):
    if not isinstance(x, torch.Tensor):
        x = torch.tensor(x, dtype=dtype)
    x = x.to(device=device, dtype=dtype)
    if x.dim() == 0:
        x = x.expand(B)
    if x.shape != (B,):
        raise ValueError(f"per-row parameter must have shape ({B},), got {tuple(x.shape)}")
    return x.contiguous()


def _out(res, name, shape, dtype, device):
    """The caller's output tensor `name` from `res` after checking it, or a new one.  The kernels
    write through raw pointers, so a buffer of the wrong shape, dtype or device, or a strided view,
    would be written out of bounds or misread: it is rejected here."""
    t = res.get(name)
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"out[{name!r}] must be a tensor")
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or t.device != device or not t.is_contiguous():
        raise ValueError(f"out[{name!r}] must be a contiguous {dtype} tensor of shape {tuple(shape)} on {device}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}"
                         + ("" if t.is_contiguous() else " (not contiguous)"))
    return t


KERNELS = {"auto": 0, "cluster": 1, "stream": 2}
MAX_TOP = 32  # TPS_MAX_TOP
MAX_HISTORY = 8192  # TPS_MAX_HISTORY


def apply_penalties(logits: torch.Tensor, history: torch.Tensor, hist_len=None, *, repetition=None,
                    frequency=None, presence=None, status: bool = False, stream=None):
    """Apply repetition, frequency and presence penalties to ``logits`` IN PLACE (the stage ahead of
    ``sample``).  For each token t that occurs c > 0 times in the row's history: z/r if z > 0 else
    z*r, then minus (frequency*c + presence), in float32 (bfloat16 logits rounded back).

    ``history``: [B, H] int32 CUDA tensor of token ids (ids outside [0, V) are ignored, so -1 pads);
    ``hist_len``: optional [B] int32 (entries past it are ignored).  ``repetition``, ``frequency``,
    ``presence``: [B] tensors or scalars, or None (off).  Returns ``logits``, or ``(logits, status)``
    when ``status`` is set (3 marks a row with invalid penalty values, which is left unchanged).
    """
    if not logits.is_cuda:
        raise ValueError("logits must be a CUDA tensor (there is no CPU path)")
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be [B, V] with unit stride along V")
    B, V = logits.shape
    ld = logits.stride(0) if B > 1 else V
    dev = logits.device
    code = _dtype_code(logits.dtype)
    if history.dim() != 2 or history.shape[0] != B or history.dtype != torch.int32:
        raise ValueError("history must be an int32 [B, H] tensor")
    if history.device != dev:
        raise ValueError("history must be on the logits' device")
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    # Every temporary (converted parameters, a contiguous copy of the history) is made on the stream
    # the kernel runs on, so it is written before the kernel reads it and its memory is not handed to
    # other work until the kernel is done with it.
    with torch.cuda.device(dev), torch.cuda.stream(s):
        h = history if history.stride(1) == 1 else history.contiguous()
        H = h.shape[1]
        ldh = h.stride(0) if B > 1 else H
        L = None if hist_len is None else _param(hist_len, B, torch.int32, dev)
        R = None if repetition is None else _param(repetition, B, torch.float32, dev)
        F = None if frequency is None else _param(frequency, B, torch.float32, dev)
        Pr = None if presence is None else _param(presence, B, torch.float32, dev)
        st = torch.empty(B, dtype=torch.int32, device=dev) if status else None
        rc = load().tps_apply_penalties(_ptr(logits), code, B, V, ld, _ptr(h), H, ldh, _ptr(L), _ptr(R), _ptr(F),
                                        _ptr(Pr), _ptr(st), ctypes.c_void_p(s.cuda_stream))
    _check(rc)
    return (logits, st) if status else logits


def sample(logits: torch.Tensor, temperature, top_k, top_p, min_p, seed, step: int = 0, *,
           want_probs: bool = False, diagnostics: bool = False, want_logprob: bool = False, top_logprobs: int = 0,
           out=None, stream=None, kernel: str = "auto"):
    """Sample one token per row of ``logits`` ([B, V] float32/bfloat16 CUDA tensor; the row stride
    may exceed V).

    Per-row parameters may be tensors of shape [B] or Python scalars: ``temperature``, ``top_p``,
    ``min_p`` (float32), ``top_k`` (int32), ``seed`` (int64, read as uint64).  ``step`` is the
    64-bit counter shared by the batch.  Returns the [B] int32 token tensor, or a dict with
    ``token``, ``status``, ``cutoff``, ``kept`` (and ``probs``) when ``diagnostics`` or
    ``want_probs`` is set.  Work is enqueued on ``stream`` (default: the current stream).
    ``kernel`` picks the sampler kernel ("auto", "cluster" or "stream"); results do not depend on it.
    ``want_logprob`` adds ``logprob``: ln P(token) under the renormalised kept distribution (0 for
    greedy rows, NaN for failed rows).  ``top_logprobs`` = n (0..32) adds ``top_idx`` and
    ``top_logprob`` ([B, n]): each row's n most probable kept tokens (probability descending, then
    index ascending) and their ln P; empty slots hold -1 and -inf, a failed row -1 and NaN.
    """
    if not logits.is_cuda:
        raise ValueError("logits must be a CUDA tensor (the sampler has no CPU path)")
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be [B, V] with unit stride along V")
    B, V = logits.shape
    ld = logits.stride(0) if B > 1 else V
    dev = logits.device
    code = _dtype_code(logits.dtype)
    n_top = int(top_logprobs)
    if not 0 <= n_top <= MAX_TOP:
        raise ValueError(f"top_logprobs must lie in [0, {MAX_TOP}]")
    if kernel not in KERNELS:
        raise ValueError(f"kernel must be one of {sorted(KERNELS)}")
    res = out if out is not None else {}
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    # Parameters converted here and outputs allocated here are made on the stream the kernel runs on
    # (see apply_penalties).
    with torch.cuda.device(dev), torch.cuda.stream(s):
        T = _param(temperature, B, torch.float32, dev)
        K = _param(top_k, B, torch.int32, dev)
        P = _param(top_p, B, torch.float32, dev)
        M = _param(min_p, B, torch.float32, dev)
        S = _param(seed, B, torch.int64, dev)
        tok = _out(res, "token", (B,), torch.int32, dev)
        probs = _out(res, "probs", (B, V), torch.float32, dev) if want_probs else None
        st = cut = kept = None
        if diagnostics:
            st = _out(res, "status", (B,), torch.int32, dev)
            cut = _out(res, "cutoff", (B,), torch.float32, dev)
            kept = _out(res, "kept", (B,), torch.int32, dev)
        lp = _out(res, "logprob", (B,), torch.float32, dev) if want_logprob else None
        ti = tl = None
        if n_top:
            ti = _out(res, "top_idx", (B, n_top), torch.int32, dev)
            tl = _out(res, "top_logprob", (B, n_top), torch.float32, dev)
        rc = load().tps_sample_full(_ptr(logits), code, B, V, ld, _ptr(T), _ptr(K), _ptr(P), _ptr(M), _ptr(S),
                                    int(step) & ((1 << 64) - 1), _ptr(tok), _ptr(probs), _ptr(st), _ptr(cut),
                                    _ptr(kept), _ptr(lp), n_top, _ptr(ti), _ptr(tl), KERNELS[kernel],
                                    ctypes.c_void_p(s.cuda_stream))
    _check(rc)
    if not (diagnostics or want_probs or want_logprob or n_top):
        return tok
    r = {"token": tok}
    if want_logprob:
        r["logprob"] = lp
    if n_top:
        r.update(top_idx=ti, top_logprob=tl)
    if diagnostics:
        r.update(status=st, cutoff=cut, kept=kept)
    if want_probs:
        r["probs"] = probs
    return r


def spec_accept(target_logits: torch.Tensor, draft_logits: torch.Tensor, target, draft, draft_token, seed,
                step: int = 0, *, diagnostics: bool = False, stream=None):
    """Speculative acceptance of one draft token per row: accept the draft's token x with
    probability min(1, P(x)/Q(x)), else draw from the normalised (P - Q)+, where P and Q are the
    renormalised kept distributions ``sample`` draws from for the target row under ``target`` and the
    draft row under ``draft`` (each a (temperature, top_k, top_p, min_p) tuple of [B] tensors or
    scalars).  ``target_logits`` and ``draft_logits``: [B, V] CUDA tensors of the same dtype and
    shape.  Returns the [B] int32 tokens, or a dict with ``token``, ``accepted`` and ``status`` when
    ``diagnostics`` is set."""
    for t in (target_logits, draft_logits):
        if not t.is_cuda or t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("logits must be [B, V] CUDA tensors with unit stride along V")
    if target_logits.shape != draft_logits.shape or target_logits.dtype != draft_logits.dtype:
        raise ValueError("target and draft logits must have the same shape and dtype")
    if target_logits.device != draft_logits.device:
        raise ValueError("target and draft logits must be on one device")
    B, V = target_logits.shape
    if B > 1 and target_logits.stride(0) != draft_logits.stride(0):
        raise ValueError("target and draft logits must share a row stride")
    ld = target_logits.stride(0) if B > 1 else V
    dev = target_logits.device
    code = _dtype_code(target_logits.dtype)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.device(dev), torch.cuda.stream(s):
        tT, tK, tP, tM = (_param(v, B, dt, dev) for v, dt in zip(target, (torch.float32, torch.int32, torch.float32,
                                                                         torch.float32)))
        dT, dK, dP, dM = (_param(v, B, dt, dev) for v, dt in zip(draft, (torch.float32, torch.int32, torch.float32,
                                                                        torch.float32)))
        X = _param(draft_token, B, torch.int32, dev)
        S = _param(seed, B, torch.int64, dev)
        tok = torch.empty(B, dtype=torch.int32, device=dev)
        acc = torch.empty(B, dtype=torch.int32, device=dev) if diagnostics else None
        st = torch.empty(B, dtype=torch.int32, device=dev) if diagnostics else None
        rc = load().tps_spec_accept(_ptr(target_logits), _ptr(draft_logits), code, B, V, ld, _ptr(tT), _ptr(tK), _ptr(tP),
                                    _ptr(tM), _ptr(dT), _ptr(dK), _ptr(dP), _ptr(dM), _ptr(X), _ptr(S),
                                    int(step) & ((1 << 64) - 1), _ptr(tok), _ptr(acc), _ptr(st),
                                    ctypes.c_void_p(s.cuda_stream))
    _check(rc)
    if not diagnostics:
        return tok
    return {"token": tok, "accepted": acc, "status": st}


def sample_rejection(logits: torch.Tensor, temperature, top_k, top_p, min_p, seed, step: int = 0, *,
                     diagnostics: bool = False, stream=None):
    """One token per row drawn by sort-free rejection rounds: the same kept set and distribution as
    ``sample``, other uniforms (``tps_sample_rejection``).  Returns the [B] int32 tokens, or a dict
    with ``token``, ``status``, ``cutoff``, ``kept`` and ``rounds`` when ``diagnostics`` is set."""
    if not logits.is_cuda or logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be a [B, V] CUDA tensor with unit stride along V")
    B, V = logits.shape
    ld = logits.stride(0) if B > 1 else V
    dev = logits.device
    code = _dtype_code(logits.dtype)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.device(dev), torch.cuda.stream(s):
        T = _param(temperature, B, torch.float32, dev)
        K = _param(top_k, B, torch.int32, dev)
        P = _param(top_p, B, torch.float32, dev)
        M = _param(min_p, B, torch.float32, dev)
        S = _param(seed, B, torch.int64, dev)
        tok = torch.empty(B, dtype=torch.int32, device=dev)
        extra = [torch.empty(B, dtype=dt, device=dev) if diagnostics else None
                 for dt in (torch.int32, torch.float32, torch.int32, torch.int32)]
        rc = load().tps_sample_rejection(_ptr(logits), code, B, V, ld, _ptr(T), _ptr(K), _ptr(P), _ptr(M), _ptr(S),
                                         int(step) & ((1 << 64) - 1), _ptr(tok), *[_ptr(x) for x in extra],
                                         ctypes.c_void_p(s.cuda_stream))
    _check(rc)
    if not diagnostics:
        return tok
    return dict(zip(("token", "status", "cutoff", "kept", "rounds"), [tok] + extra))
