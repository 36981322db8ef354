"""The C ABI library loads, exports every entry point the header declares, and rejects bad
arguments synchronously (none of these calls reaches the GPU)."""
import ctypes
import os
import re

import pytest

import nucleus_token_sampler_gb300 as tps

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tps.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tps_[a-z0-9_]+)\s*\(", text)))


def declarations():
    """name -> (return type, [parameter types]) for every function the header declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for ret, name, params in re.findall(r"([A-Za-z_][\w \*]*?)\s*\b(tps_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        ps = [q.strip() for q in params.split(",") if q.strip() and q.strip() != "void"]
        types = [re.sub(r"\s*\b\w+$", "", q) if not q.endswith("*") else q for q in ps]
        out[name] = (ret.strip(), types)
    return out


_CTYPE = {"int": ctypes.c_int, "int32_t": ctypes.c_int, "int64_t": ctypes.c_int64, "uint64_t": ctypes.c_uint64,
          "const char*": ctypes.c_char_p}


def _ctype_of(decl: str):
    d = decl.replace(" *", "*").strip()
    return ctypes.c_void_p if d.endswith("*") and d != "const char*" else _CTYPE[d]


def test_binding_signatures_match_the_header():
    """Every entry point's ctypes signature in the binding has the header's parameter count and
    types, and its return type (a mismatch would pass wrong values silently)."""
    lib = tps.load()
    decls = declarations()
    assert set(decls) == set(declared_symbols())
    for name, (ret, params) in decls.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, f"{name}: no argtypes in the binding"
        assert len(fn.argtypes) == len(params), f"{name}: {len(fn.argtypes)} argtypes, header has {len(params)}"
        for i, (have, want) in enumerate(zip(fn.argtypes, params)):
            assert have == _ctype_of(want), f"{name} parameter {i}: binding {have}, header {want!r}"
        assert fn.restype == _ctype_of(ret), f"{name}: return {fn.restype}, header {ret!r}"


def test_header_declares_entry_points():
    syms = declared_symbols()
    for s in ("tps_sample", "tps_sample_ex", "tps_max_vocab", "tps_cluster_size", "tps_status_string",
              "tps_last_cuda_error", "tps_version"):
        assert s in syms


def test_library_exports_every_declared_symbol():
    lib = tps.load()
    for s in declared_symbols():
        assert hasattr(lib, s), f"{s} declared in tps.h but not exported"


def test_version_and_status_strings():
    lib = tps.load()
    assert tps.version() >= 100
    for code in range(6):
        assert lib.tps_status_string(code)
    assert b"NaN" in lib.tps_status_string(101)
    assert lib.tps_status_string(999) == b"unknown status"


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def call(B=4, V=100, ld=None, dtype=0, logits=FAKE, T=FAKE, K=FAKE, P=FAKE, M=FAKE, S=FAKE, out=FAKE):
    lib = tps.load()
    ld = V if ld is None else ld
    v = lambda p: None if p is None else ctypes.c_void_p(p)
    return lib.tps_sample_ex(v(logits), dtype, B, V, ld, v(T), v(K), v(P), v(M), v(S), 0, v(out), None, None,
                             None, None, None)


@pytest.mark.parametrize("kw,rc", [
    (dict(B=-1), 1), (dict(V=0), 1), (dict(V=10, ld=9), 1), (dict(dtype=7), 2), (dict(dtype=-1), 2),
    (dict(logits=None), 1), (dict(T=None), 1), (dict(K=None), 1), (dict(P=None), 1), (dict(M=None), 1),
    (dict(S=None), 1), (dict(out=None), 1),
    (dict(logits=FAKE + 2), 4),
    (dict(T=FAKE + 1), 4), (dict(S=FAKE + 4), 4),
    (dict(V=1 << 20), 3),
])
def test_argument_validation(kw, rc):
    assert call(**kw) == rc


def test_empty_batch_is_a_noop():
    # B = 0 returns OK before touching any pointer or the GPU.
    assert call(B=0, logits=None, T=None, K=None, P=None, M=None, S=None, out=None) == 0


def test_kernels_per_call_rejects_bad_arguments():
    lib = tps.load()
    assert lib.tps_kernels_per_call(7, 4, 100, 0) == 0      # unknown dtype
    assert lib.tps_kernels_per_call(0, -1, 100, 0) == 0     # negative B
    assert lib.tps_kernels_per_call(0, 4, 0, 0) == 0        # empty vocabulary
    assert lib.tps_kernels_per_call(0, 4, 100, 9) == 0      # unknown kernel
    assert lib.tps_kernels_per_call(0, 0, 100, 0) == 0      # an empty batch launches nothing


def test_sample_full_checks_the_logprob_pointer():
    lib = tps.load()
    v = lambda p: None if p is None else ctypes.c_void_p(p)
    # a misaligned out_logprob is rejected before anything is launched
    def call(lp=None, n_top=0, ti=None, tl=None):
        return lib.tps_sample_full(v(FAKE), 0, 4, 100, 100, v(FAKE), v(FAKE), v(FAKE), v(FAKE), v(FAKE), 0, v(FAKE),
                                   None, None, None, None, v(lp), n_top, v(ti), v(tl), 0, None)
    assert call(lp=FAKE + 2) == 4


def test_sample_full_checks_the_top_token_arguments():
    lib = tps.load()
    v = lambda p: None if p is None else ctypes.c_void_p(p)
    def call(n_top, ti, tl):
        return lib.tps_sample_full(v(FAKE), 0, 4, 100, 100, v(FAKE), v(FAKE), v(FAKE), v(FAKE), v(FAKE), 0, v(FAKE),
                                   None, None, None, None, None, n_top, v(ti), v(tl), 0, None)
    assert call(-1, FAKE, FAKE) == 1              # negative count
    assert call(tps.MAX_TOP + 1, FAKE, FAKE) == 1  # above TPS_MAX_TOP
    assert call(3, None, FAKE) == 1               # missing index output
    assert call(3, FAKE, None) == 1               # missing log-probability output
    assert call(3, FAKE + 2, FAKE) == 4           # misaligned index output
    assert call(3, FAKE, FAKE + 1) == 4           # misaligned log-probability output


def test_apply_penalties_checks_its_arguments():
    lib = tps.load()
    v = lambda p: None if p is None else ctypes.c_void_p(p)

    def call(B=4, V=100, ld=100, hist=FAKE, H=8, ldh=8, lens=None, rep=FAKE, freq=None, pres=None, st=None,
             logits=FAKE, dtype=0):
        return lib.tps_apply_penalties(v(logits), dtype, B, V, ld, v(hist), H, ldh, v(lens), v(rep), v(freq), v(pres),
                                       v(st), None)
    assert call(H=tps.MAX_HISTORY + 1, ldh=tps.MAX_HISTORY + 1) == 1  # history too long
    assert call(H=-1) == 1                                            # negative length
    assert call(ldh=7) == 1                                           # row stride below H
    assert call(ld=99) == 1                                           # logits stride below V
    assert call(logits=None) == 1                                     # no logits
    assert call(hist=None) == 1                                       # no history with H > 0
    assert call(dtype=5) == 2                                         # unknown dtype
    assert call(logits=FAKE + 2) == 4                                 # misaligned float32 logits
    assert call(hist=FAKE + 1) == 4                                   # misaligned history
    assert call(rep=FAKE + 2) == 4                                    # misaligned penalty array
    assert call(B=0) == 0                                             # empty batch: nothing to do
    assert call(rep=None) == 0                                        # no penalty and no status: nothing to do


def test_caller_output_buffers_are_checked():
    """Output tensors a caller passes in `out` reach the kernels as raw pointers, so the binding
    rejects any whose shape, dtype, device or layout differs from what the call writes."""
    import torch
    dev = torch.device("cpu")
    ok = torch.empty(8, dtype=torch.int32)
    assert tps._out({"token": ok}, "token", (8,), torch.int32, dev) is ok
    assert tps._out({}, "token", (8,), torch.int32, dev).shape == (8,)
    bad = {
        "shape": torch.empty(7, dtype=torch.int32),
        "dtype": torch.empty(8, dtype=torch.int64),
        "strided": torch.empty(16, dtype=torch.int32)[::2],
        "2-d": torch.empty((8, 1), dtype=torch.int32),
    }
    for why, t in bad.items():
        with pytest.raises(ValueError):
            tps._out({"token": t}, "token", (8,), torch.int32, dev)
    with pytest.raises(ValueError):  # another device
        tps._out({"token": ok}, "token", (8,), torch.int32, torch.device("meta"))
    top = torch.empty((8, 4), dtype=torch.int32)  # a buffer kept from a call with fewer top tokens
    with pytest.raises(ValueError):
        tps._out({"top_idx": top}, "top_idx", (8, 8), torch.int32, dev)


def test_spec_accept_checks_its_arguments():
    lib = tps.load()
    v = lambda p: None if p is None else ctypes.c_void_p(p)

    def call(B=4, V=100, ld=100, dtype=0, zt=FAKE, zd=FAKE, tp=FAKE, dp=FAKE, x=FAKE, S=FAKE, out=FAKE, acc=None):
        return lib.tps_spec_accept(v(zt), v(zd), dtype, B, V, ld, v(tp), v(tp), v(tp), v(tp), v(dp), v(dp), v(dp),
                                   v(dp), v(x), v(S), 0, v(out), v(acc), None, None)
    assert call(B=-1) == 1 and call(V=0) == 1 and call(ld=99) == 1
    assert call(dtype=7) == 2
    assert call(B=0, zt=None, zd=None, tp=None, dp=None, x=None, S=None, out=None) == 0  # nothing to do
    for kw in ("zt", "zd", "tp", "dp", "x", "S", "out"):
        assert call(**{kw: None}) == 1, kw                     # a required pointer is missing
    assert call(zd=FAKE + 2) == 4                              # misaligned draft logits
    assert call(x=FAKE + 1) == 4                               # misaligned draft tokens
    assert call(S=FAKE + 4) == 4                               # seeds are 8-byte words
    assert call(acc=FAKE + 2) == 4                             # misaligned optional output
    assert call(V=1 << 20, ld=1 << 20) == 3                    # above the exact-mass vocabulary bound


def test_sample_rejection_checks_its_arguments():
    lib = tps.load()
    v = lambda p: None if p is None else ctypes.c_void_p(p)

    def call(B=4, V=100, ld=100, dtype=0, z=FAKE, p=FAKE, S=FAKE, out=FAKE, rounds=None):
        return lib.tps_sample_rejection(v(z), dtype, B, V, ld, v(p), v(p), v(p), v(p), v(S), 0, v(out), None, None,
                                        None, v(rounds), None)
    assert call(B=-1) == 1 and call(V=0) == 1 and call(ld=99) == 1
    assert call(dtype=3) == 2
    assert call(B=0, z=None, p=None, S=None, out=None) == 0
    for kw in ("z", "p", "S", "out"):
        assert call(**{kw: None}) == 1, kw
    assert call(z=FAKE + 2) == 4 and call(rounds=FAKE + 1) == 4
    assert call(V=1 << 20, ld=1 << 20) == 3


def test_stall_test_hook_checks_its_wait_limit():
    """The test hook takes a consumer-side wait limit of 1 ns .. 1 s; anything else is refused before
    the sampling call's own checks."""
    lib = tps.load()
    v = lambda p: None if p is None else ctypes.c_void_p(p)

    def call(wait_ns, dtype=0, B=4):
        return lib.tps_sample_stall_test(v(FAKE), dtype, B, 100, v(FAKE), v(FAKE), v(FAKE), v(FAKE), v(FAKE), 0,
                                         v(FAKE), None, 0, wait_ns, None)
    assert call(0) == 1 and call(10**9 + 1) == 1
    assert call(1000, dtype=9) == 2          # then the sampling call's checks
    assert call(1000, B=0) == 0
