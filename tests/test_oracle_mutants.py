"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Each mutant is a text edit of oracle/pa_oracle.c compiled into a temporary
library (CPU only).  A mutant that no pin rejects would mean the pins do not pin
that part of the oracle."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
from tests import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")

MUTANTS = {
    "dropped_scale": ("score[t] = scale * acc;", "score[t] = acc;"),
    "exponent_sign": ("exp(score[t] - m)", "exp(m - score[t])"),
    "no_max_shift": ("exp(score[t] - m)", "exp(score[t])"),
    "gqa_modulo_mapping": ("const int kv = h / G;", "const int kv = h % Hkv;"),
    "values_from_key_cache": ("p * elem(v_cache, dtype, row + k)", "p * elem(k_cache, dtype, row + k)"),
    "missing_normalisation": ("o[k] /= l;", "o[k] /= 1.0;"),
    "reversed_rows_in_block": ("(size_t)(t % B)) * Hkv + kv) * d;\n                double acc",
                               "(size_t)(B - 1 - t % B)) * Hkv + kv) * d;\n                double acc"),
    "query_of_kv_head": ("const size_t qoff = ((size_t)s * Hq + h) * d;",
                         "const size_t qoff = ((size_t)s * Hq + kv) * d;"),
    "one_token_short": ("for (int t = 0; t < T; ++t) {\n                const size_t phys = (size_t)block_tables[(size_t)s * max_blocks + t / B];\n                const size_t row = ((phys * B + (size_t)(t % B)) * Hkv + kv) * d;\n                const double p",
                        "for (int t = 0; t < T - 1; ++t) {\n                const size_t phys = (size_t)block_tables[(size_t)s * max_blocks + t / B];\n                const size_t row = ((phys * B + (size_t)(t % B)) * Hkv + kv) * d;\n                const double p"),
    "f16_exponent_bias": ("v = ldexp((double)(1024 + f), e - 25);", "v = ldexp((double)(1024 + f), e - 24);"),
    "f16_subnormal_scale": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "bf16_wrong_half": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b;"),
    "empty_context_not_zero": ("if (T == 0)\n                continue;", "if (T == 0)\n                { o[0] = 1.0; continue; }"),
}


def _build_mutant(tmp_path, name, old, new):
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(text.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c99", "-fopenmp", "-shared", "-fPIC", "-o", str(lib), str(path), "-lm"],
                   check=True)
    L = ctypes.CDLL(str(lib))
    L.oracle_decode.restype = ctypes.c_int
    L.oracle_decode.argtypes = oracle.lib().oracle_decode.argtypes
    L.oracle_f16_to_f64.restype = ctypes.c_double
    L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_f64.restype = ctypes.c_double
    L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    return L


def _decode_with(L):
    def dec(q, kc, vc, bt, cl, scale, dtype, hq, hkv, d, b):
        q = oracle._raw(q, dtype)
        kc = oracle._raw(kc, dtype)
        vc = oracle._raw(vc, dtype)
        bt = np.ascontiguousarray(bt, dtype=np.int32)
        cl = np.ascontiguousarray(cl, dtype=np.int32)
        out = np.zeros((cl.shape[0], hq, d))
        rc = L.oracle_decode(out.ctypes.data, q.ctypes.data, kc.ctypes.data, vc.ctypes.data,
                             oracle.DTYPE_CODE[dtype], bt.ctypes.data, bt.shape[1], cl.ctypes.data,
                             cl.shape[0], hq, hkv, d, b, kc.size // (b * hkv * d), float(scale))
        if rc != 0:
            raise ValueError(rc)
        return out
    return dec


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    L = _build_mutant(tmp_path, name, old, new)
    dec = _decode_with(L)
    caught = []
    checks = [(p.__name__, lambda p=p: p(dec)) for p in pins.ATTENTION_PINS]
    checks.append(("f16", lambda: pins.pin_f16_all_patterns(L.oracle_f16_to_f64)))
    checks.append(("bf16", lambda: pins.pin_bf16_all_patterns(L.oracle_bf16_to_f64)))
    for pname, fn in checks:
        try:
            with np.errstate(all="ignore"):
                fn()
        except Exception:
            caught.append(pname)
    assert caught, f"no pin rejects mutant {name}"


def test_unmutated_copy_passes_every_pin(tmp_path):
    L = _build_mutant(tmp_path, "identity", "double oracle_f16_to_f64", "double oracle_f16_to_f64")
    dec = _decode_with(L)
    for p in pins.ATTENTION_PINS:
        p(dec)
