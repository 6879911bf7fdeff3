"""Planted mistakes: each mutant copy of the oracle must fail at least one pin.

Every mutant is a textual edit of oracle/qmm_oracle.c (a dropped term, a wrong
sign, a wrong index, a transposed operand), compiled to a throw-away shared
library under a temporary directory.  The real oracle is never modified.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from block_quantized_gemv_gguf_gb300 import synth
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "qmm_oracle.c")

MUTANTS = {
    "q4_0_offset": ("(double)(nib - 8) * d", "(double)(nib - 7) * d"),
    "q4_0_high_nibble": ("(qs[e - 16] >> 4)", "(qs[e - 16] & 0x0f)"),
    "q8_0_index": ("(int8_t)b[2 + e]", "(int8_t)b[1 + e]"),
    "q4_k_min_sign": ("(byte >> 4);\n        out[e] = d * (double)sc * (double)q - dmin * (double)mn;",
                      "(byte >> 4);\n        out[e] = d * (double)sc * (double)q + dmin * (double)mn;"),
    "q5_k_min_sign": ("<< 4);\n        out[e] = d * (double)sc * (double)q - dmin * (double)mn;",
                      "<< 4);\n        out[e] = d * (double)sc * (double)q + dmin * (double)mn;"),
    "q4_k_scale_hi": ("((S[s - 4] >> 6) << 4)", "((S[s] >> 6) << 4)"),
    "q4_k_nibble_parity": ("int q = (s % 2 == 0) ? (byte & 0x0f)", "int q = (s % 2 == 1) ? (byte & 0x0f)"),
    "q5_k_nibble_parity": ("int lo = (s % 2 == 0) ? (byte & 0x0f)", "int lo = (s % 2 == 1) ? (byte & 0x0f)"),
    "q4_k_qs_index": ("qs[(s / 2) * 32 + e % 32]", "qs[s * 16 + e % 16]"),
    "q6_k_qh_shift": ("(qh[32 * h + l] >> (2 * j)) & 3", "(qh[32 * h + l] >> (2 * h)) & 3"),
    "q6_k_scale_index": ("sc[e / 16]", "sc[e / 32]"),
    "q6_k_offset": ("(double)(q - 32)", "(double)(q - 31)"),
    "q6_k_ql_half": ("ql[64 * h + 32 * (j % 2) + l]", "ql[64 * h + 32 * (j / 2) + l]"),
    "f16_exponent": ("ex - 25", "ex - 24"),
    "f16_subnormal": ("ldexp((double)fr, -24)", "ldexp((double)fr, -25)"),
    "matmul_x_index": ("wrow[k] * xr[k]", "wrow[k] * xr[jb->K - 1 - k]"),
    "matmul_abs_sum": ("s += fabs(p)", "s += p"),
    "row_stride": ("w + m * nb * B", "w + m * nb * (B - 1)"),
    "q8act_ties": ("rintf(blk[e] * id)", "roundf(blk[e] * id)"),
    "q8act_divisor": ("amax / 127.0f", "amax / 128.0f"),
    "q8act_scale_f16": ("scales[b] = (float)orc_f16_to_f64(orc_f32_to_f16(d));", "scales[b] = d;"),
    "q8act_nan_code": ("if (isnan(q)) q = 0.0f;", "if (isnan(q)) q = 1.0f;"),
    "q8act_id_guard": ("(d != 0.0f && isfinite(r)) ? r : 0.0f", "(d != 0.0f) ? r : 0.0f"),
    "q8act_clamp": ("q > 127.0f ? 127.0f : q", "q > 126.0f ? 126.0f : q"),
    "f16_round_even": ("nearbyint(ldexp(v, 10 - e))", "floor(ldexp(v, 10 - e))"),
    "f16_sign": ("(bits >> 16) & 0x8000u", "(bits >> 17) & 0x8000u"),
    "q5_k_qh_bit": ("int q = lo | (((qh[l] >> s) & 1) << 4);", "int q = lo | (((qh[l] >> (s / 2)) & 1) << 4);"),
    "q5_k_qs_offset": ("const uint8_t *qs = b + 48;", "const uint8_t *qs = b + 16;"),
    "q5_k_high_weight": ("int q = lo | (((qh[l] >> s) & 1) << 4);", "int q = lo | (((qh[l] >> s) & 1) << 3);"),
    "f16_subnormal_round": ("nearbyint(ldexp(v, 24))", "floor(ldexp(v, 24))"),
}


def _build_mutant(tmp, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = os.path.join(tmp, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(tmp, f"lib{name}.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    "-I", os.path.dirname(SRC), "-o", so, path, "-lm"], check=True)
    lib = ctypes.CDLL(so)
    p, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.orc_f16_to_f64.restype = ctypes.c_double
    lib.orc_dequant_block.argtypes = [ctypes.c_int, p, p]
    lib.orc_dequant.argtypes = [ctypes.c_int, p, i64, i64, p]
    lib.orc_matmul_rows.argtypes = [ctypes.c_int, p, i64, i64, p, ctypes.c_int, i64, p, i64, p, p,
                                    ctypes.c_int]
    lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
    lib.orc_f32_to_f16.restype = ctypes.c_uint16
    lib.orc_quantize_q8_0.argtypes = [p, i64, p, p]
    return lib


def _pins_fail(lib) -> list[str]:
    failed = []
    # golden blocks
    for case in pins.BLOCK_CASES:
        raw = np.frombuffer(bytes.fromhex(case["hex"]), np.uint8).copy()
        E, _ = synth.BLOCK[case["fmt"]]
        out = np.empty(E)
        lib.orc_dequant_block(case["fmt"], raw.ctypes.data, out.ctypes.data)
        exp = np.empty(E)
        for a, b, v in case["expect"]:
            exp[a:b + 1] = v
        if not np.array_equal(out, exp):
            failed.append("golden:" + case["name"])
    # f16 decoder against numpy
    h = np.arange(0, 65536, 7, dtype=np.uint16)
    ref = h.view(np.float16).astype(np.float64)
    got = np.array([lib.orc_f16_to_f64(int(v)) for v in h])
    ok = ~np.isnan(ref)
    if not np.array_equal(got[ok], ref[ok]):
        failed.append("f16")
    # brute force dequant + textbook matmul
    for fmt in (synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q6_K, synth.Q5_K):
        M, K, N = 4, 512, 2
        raw = synth.gen_weights(fmt, M, K, "mutant")
        x = synth.gen_x(N, K, "mutant")
        deq = np.empty((M, K))
        lib.orc_dequant(fmt, raw.ctypes.data, M, K, deq.ctypes.data)
        Wd = pins.brute_dequant(fmt, raw, M, K)
        if not np.array_equal(deq, Wd):
            failed.append(f"brute:{fmt}")
        Y = np.empty((N, M))
        S = np.empty((N, M))
        lib.orc_matmul_rows(fmt, raw.ctypes.data, M, K, x.ctypes.data, 0, N, None, M,
                            Y.ctypes.data, S.ctypes.data, 1)
        Yt = pins.textbook(Wd, x)
        St = (np.abs(Wd)[None] * np.abs(x.astype(np.float64))[:, None]).sum(-1)
        if not (np.all(np.abs(Y - Yt) <= 1e-12 * St) and np.allclose(S, St, rtol=1e-12)):
            failed.append(f"textbook:{fmt}")
    # activation quantizer: worked blocks and binary16 rounding against numpy
    for case in pins.Q8ACT_CASES:
        x, scale, q = pins.q8act_case_arrays(case)
        sc = np.empty(1, dtype=np.float32)
        qc = np.empty(32, dtype=np.int8)
        lib.orc_quantize_q8_0(x.ctypes.data, 32, sc.ctypes.data, qc.ctypes.data)
        if not ((sc[0] == scale or (np.isinf(scale) and np.isinf(sc[0]))) and np.array_equal(qc, q)):
            failed.append("q8act:" + case[0])
    v = pins.f16_cases()
    got = np.array([lib.orc_f32_to_f16(float(a)) for a in v], dtype=np.uint16)
    if not np.array_equal(got, pins.f16_reference_bits(v)):
        failed.append("f32_to_f16")
    return failed


@pytest.fixture(scope="module")
def tmpdir_mut():
    with tempfile.TemporaryDirectory() as d:
        yield d


def test_unmutated_copy_passes(tmpdir_mut):
    lib = _build_mutant(tmpdir_mut, "identity", "int orc_block_info", "int orc_block_info")
    assert _pins_fail(lib) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmpdir_mut, name):
    old, new = MUTANTS[name]
    lib = _build_mutant(tmpdir_mut, name, old, new)
    assert _pins_fail(lib), f"planted mistake {name} was not caught by any pin"
