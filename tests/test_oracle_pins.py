"""Pins for the oracle (CPU only).

The oracle is checked here against things other than itself:
  * the block sizes the pages state (tests/golden/block_sizes.txt);
  * hand-written worked blocks (tests/golden/blocks.txt, each with its source);
  * numpy's own binary16 decoder, for all 65536 bit patterns;
  * closed forms (constant and one-hot blocks);
  * invariants of the matmul (one-hot x, linearity, row permutation, joint
    permutation of K blocks, row subsets, bf16 inputs);
  * an independent brute-force path: a vectorised numpy dequantizer written
    separately from the format descriptions plus a textbook triple loop.
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest

import oracle
from block_quantized_gemv_gguf_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMT = {"Q8_0": oracle.Q8_0, "Q4_0": oracle.Q4_0, "Q4_K": oracle.Q4_K, "Q6_K": oracle.Q6_K, "Q5_K": oracle.Q5_K}
ALL = [oracle.Q8_0, oracle.Q4_0, oracle.Q4_K, oracle.Q6_K, oracle.Q5_K]


# --------------------------------------------------------------------------
# golden fixtures
# --------------------------------------------------------------------------
def _parse_blocks():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                name, fmt = rest.split()
                cur = dict(name=name, fmt=FMT[fmt], hex="", expect=[], cite="")
            elif key == "cite":
                cur["cite"] = rest
            elif key == "hex":
                cur["hex"] += rest.replace(" ", "")
            elif key == "expect":
                rng, val = rest.split()
                a, _, b = rng.partition("-")
                cur["expect"].append((int(a), int(b or a), float(val)))
            elif key == "end":
                cases.append(cur)
                cur = None
            else:
                raise ValueError(f"bad fixture line: {line}")
    return cases


BLOCK_CASES = _parse_blocks()


def test_block_sizes_match_pages():
    with open(os.path.join(GOLDEN, "block_sizes.txt")) as f:
        rows = [l.split()[:3] for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) == 5
    for fmt, e, b in rows:
        assert oracle.block_info(FMT[fmt]) == (int(e), int(b))


@pytest.mark.parametrize("case", BLOCK_CASES, ids=[c["name"] for c in BLOCK_CASES])
def test_golden_block(case):
    raw = bytes.fromhex(case["hex"])
    E, B = oracle.block_info(case["fmt"])
    assert len(raw) == B, f"fixture has {len(raw)} bytes, block is {B}"
    exp = np.full(E, np.nan)
    for a, b, v in case["expect"]:
        assert np.all(np.isnan(exp[a:b + 1])), "overlapping expect ranges"
        exp[a:b + 1] = v
    assert not np.any(np.isnan(exp)), "fixture does not cover every element"
    got = oracle.dequant_block(case["fmt"], raw)
    np.testing.assert_array_equal(got, exp)


def test_f16_decoder_all_bit_patterns():
    h = np.arange(65536, dtype=np.uint16)
    ref = h.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(v)) for v in h])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))  # +-0


# --------------------------------------------------------------------------
# independent brute force: numpy dequantizer + textbook triple loop
# --------------------------------------------------------------------------
def _np_f16(two_bytes: np.ndarray) -> np.ndarray:
    u = two_bytes[..., 0].astype(np.uint16) | (two_bytes[..., 1].astype(np.uint16) << 8)
    return u.view(np.float16).astype(np.float64)


def brute_dequant(fmt: int, raw: np.ndarray, M: int, K: int) -> np.ndarray:
    E, B = synth.BLOCK[fmt]
    blk = raw.reshape(M, K // E, B)
    if fmt == oracle.Q8_0:
        d = _np_f16(blk[..., 0:2])
        q = blk[..., 2:34].view(np.int8).astype(np.float64)
        w = q * d[..., None]
    elif fmt == oracle.Q4_0:
        d = _np_f16(blk[..., 0:2])
        qs = blk[..., 2:18].astype(np.int64)
        nib = np.concatenate([qs & 15, qs >> 4], axis=-1)
        w = (nib - 8).astype(np.float64) * d[..., None]
    elif fmt == oracle.Q4_K:
        d = _np_f16(blk[..., 0:2])
        dmin = _np_f16(blk[..., 2:4])
        S = blk[..., 4:16].astype(np.int64)
        sc = np.empty(S.shape[:-1] + (8,), np.int64)
        mn = np.empty_like(sc)
        sc[..., 0:4] = S[..., 0:4] % 64
        mn[..., 0:4] = S[..., 4:8] % 64
        sc[..., 4:8] = S[..., 8:12] % 16 + (S[..., 0:4] // 64) * 16
        mn[..., 4:8] = S[..., 8:12] // 16 + (S[..., 4:8] // 64) * 16
        qs = blk[..., 16:144].astype(np.int64).reshape(M, K // E, 4, 32)
        q = np.stack([qs % 16, qs // 16], axis=3).reshape(M, K // E, 8, 32)
        w = (d[..., None, None] * sc[..., None] * q - dmin[..., None, None] * mn[..., None])
        w = w.reshape(M, K // E, 256)
    elif fmt == oracle.Q5_K:
        d = _np_f16(blk[..., 0:2])
        dmin = _np_f16(blk[..., 2:4])
        S = blk[..., 4:16].astype(np.int64)
        sc = np.empty(S.shape[:-1] + (8,), np.int64)
        mn = np.empty_like(sc)
        sc[..., 0:4] = S[..., 0:4] % 64
        mn[..., 0:4] = S[..., 4:8] % 64
        sc[..., 4:8] = S[..., 8:12] % 16 + (S[..., 0:4] // 64) * 16
        mn[..., 4:8] = S[..., 8:12] // 16 + (S[..., 4:8] // 64) * 16
        qh = blk[..., 16:48].astype(np.int64)                                  # [.., 32]
        qs = blk[..., 48:176].astype(np.int64).reshape(M, K // E, 4, 32)
        lo = np.stack([qs % 16, qs // 16], axis=3).reshape(M, K // E, 8, 32)
        hi = np.stack([(qh >> s) % 2 for s in range(8)], axis=-2)              # [.., 8, 32]
        q = lo + 16 * hi
        w = (d[..., None, None] * sc[..., None] * q - dmin[..., None, None] * mn[..., None])
        w = w.reshape(M, K // E, 256)
    elif fmt == oracle.Q6_K:
        ql = blk[..., 0:128].astype(np.int64)
        qh = blk[..., 128:192].astype(np.int64)
        sc = blk[..., 192:208].view(np.int8).astype(np.float64)
        d = _np_f16(blk[..., 208:210])
        q = np.empty(blk.shape[:-1] + (256,), np.int64)
        for h in range(2):
            for j in range(4):
                src = ql[..., 64 * h + 32 * (j % 2): 64 * h + 32 * (j % 2) + 32]
                low = (src >> (4 * (j // 2))) & 15
                high = (qh[..., 32 * h: 32 * h + 32] >> (2 * j)) & 3
                q[..., 128 * h + 32 * j: 128 * h + 32 * j + 32] = low + 16 * high
        w = d[..., None] * np.repeat(sc, 16, axis=-1) * (q - 32)
    else:
        raise ValueError(fmt)
    return w.reshape(M, K)


def textbook(Wd: np.ndarray, x: np.ndarray):
    """Y[n][m] = sum_k W[m][k] x[n][k] with plain Python loops (exactly rounded sums)."""
    M, K = Wd.shape
    N = x.shape[0]
    Y = np.zeros((N, M))
    for n in range(N):
        for m in range(M):
            Y[n, m] = math.fsum(float(Wd[m, k]) * float(x[n, k]) for k in range(K))
    return Y


@pytest.mark.parametrize("fmt", ALL, ids=[synth.NAMES[f] for f in ALL])
def test_dequant_matches_brute_force(fmt):
    M, K = 8, 512
    raw = synth.gen_weights(fmt, M, K, "pin-brute")
    np.testing.assert_array_equal(oracle.dequant(fmt, raw, M, K), brute_dequant(fmt, raw, M, K))
    # One rounding to f32 (numpy's RN-even cast of the exact values).
    np.testing.assert_array_equal(oracle.dequant_f32(fmt, raw, M, K),
                                  brute_dequant(fmt, raw, M, K).astype(np.float32))


@pytest.mark.parametrize("fmt", ALL, ids=[synth.NAMES[f] for f in ALL])
def test_matmul_matches_textbook(fmt):
    M, K, N = 6, 512, 3
    raw = synth.gen_weights(fmt, M, K, "pin-textbook")
    x = synth.gen_x(N, K, "pin-textbook")
    Y, S = oracle.matmul(fmt, raw, M, K, x)
    Wd = brute_dequant(fmt, raw, M, K)
    Yt = textbook(Wd, x)
    assert np.all(np.abs(Y - Yt) <= 1e-14 * S)
    St = np.abs(Wd)[None, :, :] * np.abs(x.astype(np.float64))[:, None, :]
    np.testing.assert_allclose(S, St.sum(-1), rtol=1e-14)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
def _f16_le(v: float) -> bytes:
    return np.array([v], dtype="<f2").tobytes()


def test_q8_0_constant_block_closed_form():
    K, c = 32 * 4, -37
    d = np.float16(0.0071)
    blk = _f16_le(float(d)) + bytes([c & 0xff]) * 32
    raw = np.frombuffer(blk * (K // 32), dtype=np.uint8)
    x = synth.gen_x(2, K, "pin-q8-const")
    Y, S = oracle.matmul(oracle.Q8_0, raw, 1, K, x)
    for n in range(2):
        ref = c * float(d) * math.fsum(float(v) for v in x[n])
        assert abs(Y[n, 0] - ref) <= 1e-14 * S[n, 0]


def test_q8_0_one_hot_block():
    K, j = 64, 45
    d = np.float16(-0.0123)
    q = np.zeros(64, np.int8)
    q[j] = 1
    raw = np.frombuffer(_f16_le(float(d)) + q[:32].tobytes() + _f16_le(float(d)) + q[32:].tobytes(),
                        dtype=np.uint8)
    x = synth.gen_x(3, K, "pin-q8-onehot")
    Y, _ = oracle.matmul(oracle.Q8_0, raw, 1, K, x)
    np.testing.assert_array_equal(Y[:, 0], float(d) * x[:, j].astype(np.float64))


@pytest.mark.parametrize("q", [0, 7, 8, 15])
def test_q4_0_constant_nibble(q):
    d = np.float16(0.0042)
    raw = np.frombuffer(_f16_le(float(d)) + bytes([q | (q << 4)]) * 16, dtype=np.uint8)
    w = oracle.dequant(oracle.Q4_0, raw, 1, 32)
    assert np.all(w == (q - 8) * float(d))


def _q4k_scale_bytes(sc, mn):
    """Pack eight 6-bit (scale, min) pairs the way the GGUF reading unpacks them."""
    S = [0] * 12
    for s in range(8):
        if s < 4:
            S[s] |= sc[s] & 63
            S[s + 4] |= mn[s] & 63
        else:
            S[s + 4] |= (sc[s] & 15) | ((mn[s] & 15) << 4)
            S[s - 4] |= (sc[s] >> 4) << 6
            S[s] |= (mn[s] >> 4) << 6
    return bytes(S)


@pytest.mark.parametrize("a,b,q", [(1, 0, 3), (63, 63, 15), (40, 17, 0), (5, 60, 9)])
def test_q4_k_constant_closed_form(a, b, q):
    d, dmin = np.float16(0.0031), np.float16(0.0077)
    blk = (_f16_le(float(d)) + _f16_le(float(dmin)) + _q4k_scale_bytes([a] * 8, [b] * 8)
           + bytes([q | (q << 4)]) * 128)
    w = oracle.dequant_block(oracle.Q4_K, blk)
    assert np.all(w == float(d) * a * q - float(dmin) * b)


def test_q4_k_distinct_scales_round_trip():
    # (s+1, 2s+1) per sub-block; nibble 1 everywhere, d = 1, dmin = 1
    sc = [s + 1 for s in range(8)]
    mn = [2 * s + 1 for s in range(8)]
    blk = _f16_le(1.0) + _f16_le(1.0) + _q4k_scale_bytes(sc, mn) + bytes([0x11]) * 128
    w = oracle.dequant_block(oracle.Q4_K, blk).reshape(8, 32)
    for s in range(8):
        assert np.all(w[s] == sc[s] - mn[s])
    # The baked products d*sc and dmin*m of the pages' Q4_K repack: with
    # nibble 0 the weight is -dmin*m, with nibble 1 it is d*sc - dmin*m.
    d, dmin = np.float16(0.5), np.float16(0.25)
    blk0 = _f16_le(float(d)) + _f16_le(float(dmin)) + _q4k_scale_bytes(sc, mn) + bytes(128)
    w0 = oracle.dequant_block(oracle.Q4_K, blk0).reshape(8, 32)
    blk1 = _f16_le(float(d)) + _f16_le(float(dmin)) + _q4k_scale_bytes(sc, mn) + bytes([0x11]) * 128
    w1 = oracle.dequant_block(oracle.Q4_K, blk1).reshape(8, 32)
    for s in range(8):
        assert np.all(w0[s] == -float(dmin) * mn[s])
        assert np.all(w1[s] - w0[s] == float(d) * sc[s])


def test_q6_k_single_qh_bit_moves_one_element():
    base = bytearray(210)
    base[192:208] = bytes([1] * 16)
    base[208:210] = _f16_le(1.0)
    w0 = oracle.dequant_block(oracle.Q6_K, bytes(base))
    seen = set()
    for byte in range(64):
        for bit in range(8):
            blk = bytearray(base)
            blk[128 + byte] = 1 << bit
            w = oracle.dequant_block(oracle.Q6_K, bytes(blk))
            diff = np.nonzero(w != w0)[0]
            assert diff.size == 1
            e = int(diff[0])
            assert w[e] - w0[e] == (16 if bit % 2 == 0 else 32)
            seen.add(e)
    assert seen == set(range(256))  # every element owns exactly two qh bits


def test_q6_k_single_ql_bit_moves_one_element():
    base = bytearray(210)
    base[192:208] = bytes([1] * 16)
    base[208:210] = _f16_le(1.0)
    w0 = oracle.dequant_block(oracle.Q6_K, bytes(base))
    seen = set()
    for byte in range(128):
        for bit in range(8):
            blk = bytearray(base)
            blk[byte] = 1 << bit
            w = oracle.dequant_block(oracle.Q6_K, bytes(blk))
            diff = np.nonzero(w != w0)[0]
            assert diff.size == 1
            assert w[diff[0]] - w0[diff[0]] == 1 << (bit % 4)
            seen.add(int(diff[0]))
    assert seen == set(range(256))


# --------------------------------------------------------------------------
# matmul invariants on random blocks
# --------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", ALL, ids=[synth.NAMES[f] for f in ALL])
def test_one_hot_x_recovers_weights(fmt):
    M, K = 16, 512
    raw = synth.gen_weights(fmt, M, K, "pin-onehot")
    ks = [0, 1, 31, 32, 255, 256, 511]
    x = np.zeros((len(ks), K), np.float32)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    Y, _ = oracle.matmul(fmt, raw, M, K, x)
    Wd = oracle.dequant(fmt, raw, M, K)
    for i, k in enumerate(ks):
        np.testing.assert_array_equal(Y[i], Wd[:, k])


@pytest.mark.parametrize("fmt", ALL, ids=[synth.NAMES[f] for f in ALL])
def test_linearity(fmt):
    M, K = 12, 768
    raw = synth.gen_weights(fmt, M, K, "pin-linear")
    x1 = synth.gen_x(2, K, "pin-linear-1")
    x2 = synth.gen_x(2, K, "pin-linear-2")
    x1[:, 1::2] = 0.0  # disjoint supports and power-of-two weights keep the
    x2[:, 0::2] = 0.0  # combination a*x1 + b*x2 exact in f32
    a, b = 0.5, -2.0
    Y1, S1 = oracle.matmul(fmt, raw, M, K, x1)
    Y2, S2 = oracle.matmul(fmt, raw, M, K, x2)
    Y12, _ = oracle.matmul(fmt, raw, M, K, (a * x1 + b * x2).astype(np.float32))
    assert np.all(np.abs(Y12 - (a * Y1 + b * Y2)) <= 1e-13 * (abs(a) * S1 + abs(b) * S2))


@pytest.mark.parametrize("fmt", ALL, ids=[synth.NAMES[f] for f in ALL])
def test_row_permutation(fmt):
    M, K = 10, 512
    E, B = synth.BLOCK[fmt]
    rb = K // E * B
    raw = synth.gen_weights(fmt, M, K, "pin-perm")
    perm = np.random.default_rng(1).permutation(M)
    rawp = raw.reshape(M, rb)[perm].reshape(-1)
    x = synth.gen_x(3, K, "pin-perm")
    Y, _ = oracle.matmul(fmt, raw, M, K, x)
    Yp, _ = oracle.matmul(fmt, rawp, M, K, x)
    np.testing.assert_array_equal(Yp, Y[:, perm])


@pytest.mark.parametrize("fmt", ALL, ids=[synth.NAMES[f] for f in ALL])
def test_joint_k_block_permutation(fmt):
    M, K = 6, 1024
    E, B = synth.BLOCK[fmt]
    nb = K // E
    raw = synth.gen_weights(fmt, M, K, "pin-kperm")
    x = synth.gen_x(2, K, "pin-kperm")
    perm = np.random.default_rng(2).permutation(nb)
    rawp = raw.reshape(M, nb, B)[:, perm].reshape(-1)
    xp = x.reshape(2, nb, E)[:, perm].reshape(2, K)
    Y, S = oracle.matmul(fmt, raw, M, K, x)
    Yp, _ = oracle.matmul(fmt, rawp, M, K, xp)
    assert np.all(np.abs(Y - Yp) <= 1e-13 * S)


def test_row_subset_and_threads():
    fmt, M, K = oracle.Q4_K, 40, 512
    raw = synth.gen_weights(fmt, M, K, "pin-rows")
    x = synth.gen_x(4, K, "pin-rows")
    Y, S = oracle.matmul(fmt, raw, M, K, x, nthreads=1)
    Y3, S3 = oracle.matmul(fmt, raw, M, K, x, nthreads=3)
    np.testing.assert_array_equal(Y, Y3)
    rows = np.array([39, 0, 17, 17, 5])
    Yr, Sr = oracle.matmul(fmt, raw, M, K, x, rows=rows)
    np.testing.assert_array_equal(Yr, Y[:, rows])
    np.testing.assert_array_equal(Sr, S[:, rows])
    assert np.all(S >= np.abs(Y))


def test_bf16_x_equals_expanded_f32():
    fmt, M, K = oracle.Q6_K, 8, 512
    raw = synth.gen_weights(fmt, M, K, "pin-bf16")
    x = synth.gen_x(3, K, "pin-bf16")
    xb = synth.f32_to_bf16_bits(x)
    Yb, Sb = oracle.matmul(fmt, raw, M, K, xb)
    Yf, Sf = oracle.matmul(fmt, raw, M, K, synth.bf16_bits_to_f32(xb))
    np.testing.assert_array_equal(Yb, Yf)
    np.testing.assert_array_equal(Sb, Sf)


def test_bad_arguments_rejected():
    raw = np.zeros(18, np.uint8)
    with pytest.raises(ValueError):
        oracle.dequant(oracle.Q4_0, raw, 1, 31)          # K not a multiple of 32
    with pytest.raises(ValueError):
        oracle.matmul(oracle.Q4_0, raw, 1, 32, np.zeros((1, 32), np.float32), rows=[1])
    with pytest.raises(ValueError):
        oracle.block_info(7)


def test_tolerance_helper():
    Y = np.array([[1.0, -2.0]])
    S = np.array([[10.0, 10.0]])
    ok, _ = oracle.within(np.array([[1.00009, -2.0]]), Y, S, 1e-5, 1e-6)
    assert ok
    ok, _ = oracle.within(np.array([[1.0002, -2.0]]), Y, S, 1e-5, 1e-6)
    assert not ok


# ---------------------------------------------------------------------------
# Q8_0 activation quantizer ("cera 0.5.2 src/backend/cpu.rs",
# quantize_f32_to_q8_0_scalar): scale amax/127 in float, rounded through
# binary16; codes rint(x * (1/d)) with ties to even, clamped, NaN -> 0.
# Worked blocks with closed-form results: (name, {index: x}, scale, {index: code}).
# ---------------------------------------------------------------------------
_D127 = float(np.float32(1.0) / np.float32(127.0))
Q8ACT_CASES = [
    # amax 127 -> d = 1 exactly, id = 1: codes are x rounded half to even
    ("unit_scale_ties", {0: 127.0, 1: 2.5, 2: 3.5, 3: -2.5, 4: -127.0, 5: 0.5, 6: 1.5, 7: -0.5},
     1.0, {0: 127, 1: 2, 2: 4, 3: -2, 4: -127, 5: 0, 6: 2, 7: 0}),
    # amax 1 -> d = fl(1/127); 1/d rounds to 127 exactly; x = 0.5 is a tie (63.5 -> 64);
    # the binary16 scale is 2^-7 (1 + 8/1024)
    ("unit_amax", {0: 1.0, 1: 0.5, 2: -0.25, 3: 0.75}, 2.0 ** -7 * (1 + 8 / 1024),
     {0: 127, 1: 64, 2: -32, 3: 95}),
    ("zero_block", {}, 0.0, {}),
    # a NaN element is skipped by the max fold and gets code 0
    ("nan_element", {0: 127.0, 1: float("nan"), 2: 5.0}, 1.0, {0: 127, 1: 0, 2: 5}),
    # amax = inf: d = inf, 1/d = 0 is finite, so id = 0 and every code is 0;
    # the scale stays infinite
    ("inf_element", {0: float("inf"), 1: 3.0}, float("inf"), {0: 0, 1: 0}),
    # subnormal amax: 1/d overflows, id = 0; d underflows binary16 to 0
    ("subnormal_amax", {0: 1e-40, 1: -5e-41}, 0.0, {0: 0, 1: 0}),
    # d = 70000 overflows binary16 (scale inf) but the codes use the float d
    ("f16_overflow_scale", {0: 127.0 * 70000.0, 1: 70000.0, 2: -35000.0}, float("inf"),
     {0: 127, 1: 1, 2: 0}),
]


def q8act_case_arrays(case):
    name, xs, scale, codes = case
    x = np.zeros(32, dtype=np.float32)
    for i, v in xs.items():
        x[i] = v
    q = np.zeros(32, dtype=np.int8)
    for i, v in codes.items():
        q[i] = v
    return x, np.float32(scale), q


@pytest.mark.parametrize("case", Q8ACT_CASES, ids=[c[0] for c in Q8ACT_CASES])
def test_q8_0_act_worked_blocks(case):
    x, scale, q = q8act_case_arrays(case)
    s, c = oracle.quantize_q8_0(x)
    assert s.shape == (1,) and c.shape == (32,)
    assert s[0] == scale or (np.isinf(scale) and np.isinf(s[0])), (s[0], scale)
    assert np.array_equal(c, q), c


def test_q8_0_act_unit_amax_reciprocal_is_exact():
    # the reading of the worked block above: fl(1 / fl(1/127)) == 127
    assert np.float32(1.0) / np.float32(_D127) == np.float32(127.0)


def f16_reference_bits(v: np.ndarray) -> np.ndarray:
    """numpy's float32 -> float16 cast (round to nearest even) as bit patterns."""
    with np.errstate(over="ignore"):
        return v.astype(np.float16).view(np.uint16)


def f16_cases() -> np.ndarray:
    rng = np.random.default_rng(20261202)
    parts = [
        rng.standard_normal(3000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 3000),
        np.float32(2.0) ** np.arange(-30, 17, dtype=np.float32),
        # exact ties of binary16 rounding: odd multiples of half a unit in the last place
        ((np.arange(1, 400, 2, dtype=np.float64) / 2 + 1024) * 2.0 ** -10).astype(np.float32),
        ((np.arange(1, 200, 2, dtype=np.float64) / 2) * 2.0 ** -24).astype(np.float32),   # subnormal ties
        np.array([65504, 65519, 65519.998, 65520, 65536, 1e9, 6.1e-5, 6.097555e-05, 5.96e-8, 2.98e-8,
                  2.9802322e-08, 2.99e-8, 0.0, -0.0, np.inf, -np.inf], dtype=np.float32),
    ]
    v = np.concatenate(parts).astype(np.float32)
    return np.concatenate([v, -v])


def test_f32_to_f16_matches_numpy():
    v = f16_cases()
    got = np.array([oracle.f32_to_f16(float(a)) for a in v], dtype=np.uint16)
    assert np.array_equal(got, f16_reference_bits(v))
    assert (oracle.f32_to_f16(float("nan")) & 0x7c00) == 0x7c00 and (oracle.f32_to_f16(float("nan")) & 0x3ff)


def q8act_numpy(x: np.ndarray):
    """Independent float32 restatement with numpy's own binary16 cast."""
    b = x.astype(np.float32).reshape(-1, 32)
    amax = np.fmax.reduce(np.abs(b), axis=1, initial=np.float32(0))
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        d = (amax / np.float32(127)).astype(np.float32)
        r = (np.float32(1) / d).astype(np.float32)
        idv = np.where((d != 0) & np.isfinite(r), r, np.float32(0)).astype(np.float32)
        q = np.rint((b * idv[:, None]).astype(np.float32))
        q = np.where(np.isnan(q), 0, np.clip(q, -128, 127)).astype(np.int8)
        s = d.astype(np.float16).astype(np.float32)
    return s, q.reshape(x.shape)


def test_q8_0_act_random_blocks_match_numpy():
    x = synth.gen_x(8, 1024, "q8act-pin")
    x[0, :32] *= np.float32(1e-3)
    x[1, 32:64] *= np.float32(3e4)
    s, q = oracle.quantize_q8_0(x)
    s2, q2 = q8act_numpy(x.reshape(-1))
    assert np.array_equal(s.reshape(-1), s2) and np.array_equal(q.reshape(-1), q2.reshape(-1))


def test_q8act_matmul_one_hot_closed_form():
    # X = c * e_k: the block of k has amax c, so its code at k is 127 and
    # y[m] = w(m, k) * 127 * f16(c / 127)
    fmt, M, K, k, c = synth.Q4_0, 8, 256, 77, np.float32(3.0)
    w = synth.gen_weights(fmt, M, K, "q8act-onehot")
    x = np.zeros((1, K), dtype=np.float32)
    x[0, k] = c
    Y, S = oracle.matmul_q8act(fmt, w, M, K, x)
    scale = np.float64(np.float32(c / np.float32(127)).astype(np.float16))
    Wd = oracle.dequant(fmt, w, M, K)
    assert np.array_equal(Y[0], Wd[:, k] * 127 * scale)
    assert np.array_equal(S[0], np.abs(Y[0]))


def test_q8act_bad_length_rejected():
    with pytest.raises(ValueError):
        oracle.quantize_q8_0(np.zeros(31, dtype=np.float32))


@pytest.mark.parametrize("a,b,q,h", [(1, 0, 0, 0), (5, 3, 7, 1), (63, 63, 15, 1), (17, 40, 9, 0)])
def test_q5_k_constant_closed_form(a, b, q, h):
    # every nibble q, every qh bit h: w = d*a*(q + 16h) - dmin*b
    d, dmin = np.float16(0.0031), np.float16(0.0077)
    blk = (_f16_le(float(d)) + _f16_le(float(dmin)) + _q4k_scale_bytes([a] * 8, [b] * 8)
           + bytes([0xFF if h else 0]) * 32 + bytes([q | (q << 4)]) * 128)
    w = oracle.dequant_block(oracle.Q5_K, blk)
    assert np.all(w == float(d) * a * (q + 16 * h) - float(dmin) * b)


def test_q5_k_single_qh_bit_moves_one_element():
    # bit s of qh[l] is bit 4 of element 32 s + l, and nothing else
    base = bytearray(176)
    base[0:2] = _f16_le(1.0)
    base[4:16] = _q4k_scale_bytes([1] * 8, [0] * 8)
    w0 = oracle.dequant_block(oracle.Q5_K, bytes(base))
    for l in range(32):
        for s in range(8):
            blk = bytearray(base)
            blk[16 + l] = 1 << s
            w = oracle.dequant_block(oracle.Q5_K, bytes(blk))
            diff = np.nonzero(w != w0)[0]
            assert list(diff) == [32 * s + l]
            assert w[32 * s + l] - w0[32 * s + l] == 16


def test_swiglu_against_library_sigmoid():
    # silu(g) * u against scipy's logistic function, over a wide range of g
    special = pytest.importorskip("scipy.special")
    g = np.concatenate([np.linspace(-60, 60, 241), [0.0, -1e-8, 1e-8, 700.0, -700.0]])
    u = np.linspace(-3, 3, g.size)
    out, _ = oracle.swiglu(g, np.zeros_like(g), u, np.zeros_like(u), 0.0, 0.0)
    ref = g * special.expit(g) * u
    assert np.allclose(out, ref, rtol=1e-14, atol=1e-300)
    assert out[g.size - 2] == 700.0 * u[g.size - 2]          # sigmoid(700) == 1 in double


def test_swiglu_bound_covers_perturbations():
    # the first-order bound holds for worst-case perturbations of g and u
    rng = np.random.default_rng(3)
    g = rng.normal(0, 4, 2000)
    u = rng.normal(0, 2, 2000)
    S = np.abs(rng.normal(0, 30, 2000))
    out, bound = oracle.swiglu(g, S, u, S, 1e-5, 1e-6)
    e = 1e-5 * S + 1e-6
    for sg in (-1, 1):
        for su in (-1, 1):
            p, _ = oracle.swiglu(g + sg * e, S, u + su * e, S, 0.0, 0.0)
            assert np.all(np.abs(p - out) <= bound)
