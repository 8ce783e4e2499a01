"""Pins of the CPU oracle to facts other than its own code.

Each test cites what fixes the expected values: a value worked out by hand
from a printed formula, a closed form, an invariant of the mathematics, a
published known-answer vector, or a library routine (libc memcpy via Python
slicing, IEEE arithmetic via numpy float64) computed independently.
"""
import numpy as np
import pytest

import oracle


# ---------------------------------------------------------------------------
# PrepSrcValue - "TransferBench data validation", "Expected source pattern"
# ---------------------------------------------------------------------------
def test_prep_src_value_hand_worked(golden):
    for buf, i, v in golden("prep_src_value.txt"):
        assert oracle.prep_src_value(int(buf), int(i)) == float(v), (buf, i)


@pytest.mark.parametrize("k", [0, 1, 2, 7])
@pytest.mark.parametrize("start", [0, 383 * 5 + 17, 2**33 + 5, 2**40 + 123])
def test_prep_src_value_window_is_permutation(k, start):
    # 383 is prime and 517 = 134 (mod 383) is invertible, so i -> (517 i) % 383
    # permutes the residues: any 383 consecutive indices give {31..413}*(k+1),
    # whose sum is 85,026*(k+1).  Large starts catch 32-bit index overflow.
    vals = np.array([oracle.prep_src_value(k, start + j) for j in range(383)])
    assert sorted(vals.tolist()) == [float(v * (k + 1)) for v in range(31, 414)]
    assert vals.sum() == 85026 * (k + 1)


def test_prep_src_value_period_and_vector_form():
    n = 383 * 3 + 11
    for k in range(3):
        ref = oracle.prepare_reference(n, k)
        assert ref.dtype == np.float32 and ref.size == n
        assert np.array_equal(ref[:383], ref[383:766])
        assert ref[5] == oracle.prep_src_value(k, 5)
        assert ref.max() == 413 * (k + 1) and ref.min() == 31 * (k + 1)


# ---------------------------------------------------------------------------
# dstReference - "Expected destination (dstReference)" and the table
# "Number of sources / Expected value"
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("nsrc", [1, 2, 3, 5, 8])
def test_dst_reference_closed_form_default_pattern(nsrc):
    # src_k[i] = (k+1) * P(i) with P(i) = PrepSrcValue(0, i), so
    # sum_k src_k[i] = N(N+1)/2 * P(i), an integer below 2^24 and therefore
    # exact in float32 whatever the order of the adds.
    n = 4096 + 7
    srcs = [oracle.prepare_reference(n, k) for k in range(nsrc)]
    got = oracle.dst_reference(srcs)
    base = oracle.prepare_reference(n, 0).astype(np.int64)
    expect = (base * (nsrc * (nsrc + 1) // 2)).astype(np.float32)
    assert np.array_equal(got, expect)


def test_dst_reference_three_source_values():
    # 3 sources of the default pattern: dst = 6 * P(i); P(0..3) = 31,165,299,50.
    srcs = [oracle.prepare_reference(4, k) for k in range(3)]
    assert oracle.dst_reference(srcs).tolist() == [186.0, 990.0, 1794.0, 300.0]


@pytest.mark.parametrize("byte", [0x00, 0xA5, 0xFF])
def test_dst_reference_zero_sources_is_memset(byte):
    got = oracle.dst_reference([], n=33, memset_byte=byte)
    assert np.all(got.view(np.uint8) == byte)


def test_dst_reference_one_source_is_a_bit_copy():
    # dst[i] == src0[i]: the bytes themselves, including -0.0, NaN payloads,
    # signalling NaNs, infinities and subnormals.
    bits = np.array([0x80000000, 0x7FC00001, 0xFF800001, 0x7FA00000, 0x00000001, 0x807FFFFF,
                     0x7F800000, 0xFF800000, 0x3F800000], dtype=np.uint32)
    got = oracle.dst_reference([bits.view(np.float32)])
    assert np.array_equal(got.view(np.uint32), bits)


def test_dst_reference_adds_left_to_right():
    # 1 + 2^-24 is a tie that rounds to even (1.0); doing it twice stays 1.0.
    # The other association, 1 + (2^-24 + 2^-24), would give 1 + 2^-23.
    one = np.array([1.0], np.float32)
    eps = np.array([2.0**-24], np.float32)
    assert oracle.dst_reference([one, eps, eps])[0] == np.float32(1.0)
    assert oracle.dst_reference([eps, eps, one])[0] == np.float32(1.0 + 2.0**-23)


def _finite_random_floats(g, n):
    bits = g.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    bits &= ~np.uint32(0x7F800000) | np.uint32(0x7F000000)  # exponent never all-ones
    # sprinkle subnormals, zeros of both signs and values close to each other
    bits[::7] &= np.uint32(0x807FFFFF)
    bits[::11] = np.uint32(0x80000000)
    return bits.view(np.float32)


@pytest.mark.parametrize("nsrc", [2, 3, 4, 6])
def test_dst_reference_matches_ieee_binary32_steps(nsrc):
    # Each step must be one binary32 round-to-nearest-even add.  Reference:
    # the exact sum of two float32 values rounded once to binary64 and then to
    # binary32; double rounding is innocuous for a single add since
    # 53 >= 2*24 + 2 (Figueroa, "When is double rounding innocuous?", 1995).
    g = np.random.default_rng(1000 + nsrc)
    n = 20000
    srcs = [_finite_random_floats(g, n) for _ in range(nsrc)]
    # Scale half the elements so that operands often share an exponent range
    # and cancel, while the other half spans the whole range.
    for s in srcs[1:]:
        near = srcs[0][: n // 2].astype(np.float64) * -g.uniform(0.5, 2.0, n // 2)
        s[: n // 2] = np.clip(near, -3.0e38, 3.0e38).astype(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        acc = srcs[0].copy()
        for s in srcs[1:]:
            acc = (acc.astype(np.float64) + s.astype(np.float64)).astype(np.float32)
    got = oracle.dst_reference(srcs)
    assert np.array_equal(got.view(np.uint32), acc.view(np.uint32))


def test_dst_reference_ieee_special_cases():
    a = np.array([1.5, -0.0, 2.0**-149, 3.0e38, -7.25], np.float32)
    b = np.array([-1.5, -0.0, 2.0**-149, 3.0e38, 0.0], np.float32)
    got = oracle.dst_reference([a, b])
    assert got[0] == 0.0 and not np.signbit(got[0])      # x + (-x) = +0
    assert got[1] == 0.0 and np.signbit(got[1])          # -0 + -0 = -0
    assert got[2] == np.float32(2.0**-148)               # subnormals kept, no flush
    assert np.isinf(got[3]) and got[3] > 0               # overflow to +inf
    assert got[4] == np.float32(-7.25)                   # x + 0 = x


# ---------------------------------------------------------------------------
# fillPattern and fillCompress - "Expected source pattern"
# ---------------------------------------------------------------------------
def test_fill_pattern_repeats_the_vector():
    pat = np.array([1.5, -2.0, 3.25], np.float32)
    got = oracle.fill_pattern(100, pat)
    assert np.array_equal(got, np.resize(pat, 100))
    # written out by hand: the vector, again, then its start
    assert got[:7].tolist() == [1.5, -2.0, 3.25, 1.5, -2.0, 3.25, 1.5]


def test_fill_pattern_edges():
    # one value: a constant buffer; a vector longer than the buffer: its
    # first n values; n = 0: nothing; values kept bit for bit (-0, subnormal)
    assert oracle.fill_pattern(5, [7.0]).tolist() == [7.0] * 5
    assert oracle.fill_pattern(2, [4.0, 5.0, 6.0]).tolist() == [4.0, 5.0]
    assert oracle.fill_pattern(0, [1.0]).size == 0
    odd = np.array([-0.0, np.float32(1e-45), np.inf], np.float32)
    got = oracle.fill_pattern(6, odd)
    assert np.array_equal(got.view(np.uint32), np.tile(odd.view(np.uint32), 2))
    with pytest.raises(ValueError):
        oracle.fill_pattern(4, [])


def test_splitmix64_known_answers(golden):
    rows = golden("splitmix64.txt")
    kat = [r for r in rows if r[0] != "counts"]
    seed = int(kat[0][0])
    stream = oracle.splitmix64_stream(seed, len(kat))
    for s, idx, val in kat:
        assert int(stream[int(idx)]) == int(val)
    counts = [r for r in rows if r[0] == "counts"]
    s = oracle.splitmix64_stream(int(counts[0][1]), 100000)
    f = (s >> np.uint64(11)).astype(np.float64) * 2.0**-53
    hist = np.bincount(np.floor(f * 5).astype(int), minlength=5)
    for _, _, cls, cnt in counts:
        assert hist[int(cls)] == int(cnt)


def _compress_expectation(n, pct, seed, k):
    """Independent numpy restatement of the fillCompress reading: draws
    17L..17L+16 of the stream seeded with seed + k, mode from the first,
    floats from the rest, zero every odd aligned chunk of the mode's size."""
    lines = (n + 15) // 16
    s = oracle.splitmix64_stream(seed + k, 17 * lines).reshape(lines, 17)
    r = (s[:, 0] % np.uint64(100)).astype(np.int64)
    cum = np.cumsum(pct)
    mode = np.searchsorted(cum, r, side="right")
    vals = ((s[:, 1:] >> np.uint64(40)).astype(np.float64) * 2.0**-23 - 1.0).astype(np.float32)
    raw = vals.copy().view(np.uint8).reshape(lines, 64)
    byte = np.arange(64)
    for m, chunk in ((1, 1), (2, 2), (3, 4), (4, 32)):
        rows = mode == m
        raw[np.ix_(rows, (byte // chunk) % 2 == 1)] = 0
    return raw.view(np.float32).reshape(-1)[:n], mode, vals


@pytest.mark.parametrize("n,pct,k", [(16 * 4000, (40, 20, 0, 20, 20), 0),
                                     (16 * 1000 + 5, (20, 20, 20, 20, 20), 1),
                                     (16 * 500, (100, 0, 0, 0, 0), 2)])
def test_fill_compress_structure(n, pct, k):
    seed = 0x5EED
    got = oracle.fill_compress(n, pct, seed, k)
    exp, mode, vals = _compress_expectation(n, pct, seed, k)
    assert np.array_equal(got.view(np.uint32), exp.view(np.uint32))
    # Unmasked floats lie in [-1, 1) on the 2^-23 grid.
    assert vals.min() >= -1.0 and vals.max() < 1.0
    assert np.all(np.floor(vals.astype(np.float64) * 2**23) == vals.astype(np.float64) * 2**23)
    # Modes with 0% never occur; the others stay within 6 sigma of their share.
    cnt = np.bincount(mode, minlength=5)
    lines = mode.size
    for m in range(5):
        p = pct[m] / 100.0
        if p == 0:
            assert cnt[m] == 0
        else:
            assert abs(cnt[m] - p * lines) <= 6 * np.sqrt(lines * p * (1 - p)) + 1


def test_fill_compress_zero_masks_by_mode():
    # Per mode, where the zero bytes of a line sit (bytes of 16 floats, in
    # little-endian memory order): 1B0 odd bytes, 2B0 odd byte pairs, 4B0 odd
    # floats, 32B0 the upper half.
    got = oracle.fill_compress(16 * 3000, (0, 25, 25, 25, 25), 7, 0)
    raw = got.view(np.uint8).reshape(-1, 64)
    _, mode, _ = _compress_expectation(16 * 3000, (0, 25, 25, 25, 25), 7, 0)
    b = np.arange(64)
    masks = {1: b % 2 == 1, 2: (b // 2) % 2 == 1, 3: (b // 4) % 2 == 1, 4: b >= 32}
    for m, zero in masks.items():
        rows = raw[mode == m]
        assert rows.shape[0] > 500
        assert np.all(rows[:, zero] == 0)
        # the kept bytes are not all zero (random floats rarely have zero bytes)
        assert np.mean(rows[:, ~zero] != 0) > 0.9


def _golden_compress_cases(golden):
    rows = golden("fill_compress.txt")
    cases = {}
    for r in rows:
        if r[0] == "case":
            name, seed, k, n = r[1], int(r[2]), int(r[3]), int(r[4])
            pct = tuple(int(x) for x in r[5:10])
            modes = [int(x) for x in r[10:]]
            cases[name] = dict(seed=seed, k=k, n=n, pct=pct, modes=modes, words={})
        elif r[0] == "word":
            cases[r[1]]["words"][int(r[2])] = int(r[3], 16)
    return rows, cases


def test_fill_compress_golden_draws_are_the_published_vector(golden):
    # The golden file's stream for seed 1234567 starts with the published
    # SplitMix64 known-answer vector, so its words rest on that vector and
    # not on the oracle's generator.
    rows, _ = _golden_compress_cases(golden)
    draws = {int(r[2]): int(r[3]) for r in rows if r[0] == "draw"}
    kat = [r for r in golden("splitmix64.txt") if r[0] != "counts"]
    for seed, idx, val in kat:
        assert seed == "1234567" and draws[int(idx)] == int(val)
    for i, v in draws.items():
        row = next(r for r in rows if r[0] == "draw" and int(r[2]) == i)
        assert int(row[4]) == v % 100 and int(row[5]) == v >> 40


def test_fill_compress_hand_worked_golden(golden):
    # "Expected source pattern", fillCompress row, under the reading stated in
    # the oracle: every word of tests/golden/fill_compress.txt (mode draw,
    # float mapping, each zero mask, a partial last line, seed + k).
    _, cases = _golden_compress_cases(golden)
    assert len(cases) == 8
    seen_modes = set()
    for name, c in cases.items():
        got = oracle.fill_compress(c["n"], c["pct"], c["seed"], c["k"]).view(np.uint32)
        want = np.array([c["words"][i] for i in range(c["n"])], dtype=np.uint32)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, f"{name}: word {bad[0]} {got[bad[0]]:08X} != {want[bad[0]]:08X}"
        seen_modes.update(c["modes"][: (c["n"] + 15) // 16])
    assert seen_modes == {0, 1, 2, 3, 4}


# Slips a restatement of fillCompress could plausibly make, planted one at a
# time into a copy of oracle.c: (what it gets wrong, text replaced, replacement).
_MODE_BLOCK = ("        uint64_t r = orc_splitmix64_next(&state) % 100u;\n"
               "        int mode = 0;\n"
               "        while (mode < 4 && r >= cum[mode])\n"
               "            ++mode;\n")
_FLOAT_LOOP_END = ("            vals[j] = (float)(int32_t)(d >> 40) * 0x1p-23f - 1.0f;\n"
                   "        }\n")
_SLIPS = [
    ("mode drawn after the floats", _MODE_BLOCK + "\n        float vals[16];\n",
     "        float vals[16];\n"),
    ("shift by 41", "(d >> 40)", "(d >> 41)"),
    ("low 24 bits", "(d >> 40)", "(d & 0xFFFFFFu)"),
    ("no -1 offset", "* 0x1p-23f - 1.0f", "* 0x1p-23f"),
    ("seed xor k", "seed + (uint64_t)bufferIdx", "seed ^ (uint64_t)bufferIdx"),
    ("k ignored", "seed + (uint64_t)bufferIdx", "seed"),
    ("mode boundary <=", "r >= cum[mode]", "r > cum[mode]"),
    ("even chunks zeroed", "(b / chunk) % 2u == 1u", "(b / chunk) % 2u == 0u"),
    ("big-endian bytes", "bytes[b] = 0;", "bytes[63u - b] = 0;"),
    ("32B0 as 16-byte chunks", "{ 0u, 1u, 2u, 4u, 32u }", "{ 0u, 1u, 2u, 4u, 16u }"),
    ("2B0 as 4B0", "{ 0u, 1u, 2u, 4u, 32u }", "{ 0u, 1u, 4u, 4u, 32u }"),
    ("partial line dropped", "uint64_t nLines = (n + 15u) / 16u;", "uint64_t nLines = n / 16u;"),
]


def test_fill_compress_golden_catches_planted_slips(golden, tmp_path):
    # Mutation check of the pin above: each slip, compiled into its own copy
    # of the oracle on the CPU, must change at least one golden word.
    import ctypes
    import subprocess
    from oracle import _build
    src = open(_build.SRC).read()
    _, cases = _golden_compress_cases(golden)
    for i, (what, old, new) in enumerate(_SLIPS):
        if what == "mode drawn after the floats":
            assert old in src and _FLOAT_LOOP_END in src, what
            mutated = src.replace(old, new).replace(_FLOAT_LOOP_END, _FLOAT_LOOP_END + _MODE_BLOCK)
        else:
            assert old in src, what
            mutated = src.replace(old, new)
        c_file = tmp_path / f"slip{i}.c"
        so_file = tmp_path / f"slip{i}.so"
        c_file.write_text(mutated)
        flags = [f for f in _build.CFLAGS if f != "-Werror"]
        subprocess.run(["gcc", *flags, str(c_file), "-o", str(so_file)], check=True)
        lib = ctypes.CDLL(str(so_file))
        lib.orc_fill_compress.restype = ctypes.c_int
        lib.orc_fill_compress.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p,
                                          ctypes.c_uint64, ctypes.c_int64]
        caught = False
        for c in cases.values():
            out = np.full(c["n"], 0xA5A5A5A5, dtype=np.uint32)
            pct = np.array(c["pct"], dtype=np.uint32)
            lib.orc_fill_compress(out.ctypes.data, c["n"], pct.ctypes.data, c["seed"], c["k"])
            want = np.array([c["words"][j] for j in range(c["n"])], dtype=np.uint32)
            if not np.array_equal(out, want):
                caught = True
                break
        assert caught, f"the golden words do not catch: {what}"


def test_fill_compress_rejects_bad_percentages():
    with pytest.raises(ValueError):
        oracle.fill_compress(16, (50, 20, 0, 20, 20), 1)


# ---------------------------------------------------------------------------
# Rotation - PR #365 "Technical Details" and "Test Result"
# ---------------------------------------------------------------------------
def test_rotation_plan_pinned_examples(golden):
    for nb, rb, off, k, alloc in golden("rotation.txt"):
        K, stride, a = oracle.rotation_plan(int(nb), int(rb), int(off))
        assert (K, a) == (int(k), int(alloc))


@pytest.mark.parametrize("mib,K", [(8, 32), (16, 16), (32, 8), (64, 4), (128, 2), (256, 1),
                                   (512, 1)])
def test_rotation_plan_sweep_sizes(mib, K):
    nb = mib << 20
    k, stride, alloc = oracle.rotation_plan(nb, 256 << 20)
    assert k == K and stride == nb and alloc == K * nb          # K * numBytes
    assert oracle.rotation_plan(nb, 0) == (1, nb, nb)            # 0 disables


def test_rotation_plan_offset_stride_and_errors():
    assert oracle.rotation_plan(4 << 20, 256 << 20, 64)[2] == (256 << 20) + 64
    # ceil: 10 MiB of rotation over 3 MiB transfers needs 4 slices
    assert oracle.rotation_plan(3 << 20, 10 << 20)[0] == 4
    # a stride keeps 256-byte alignment; the last slice needs only numBytes
    k, stride, alloc = oracle.rotation_plan(1000, 4000)
    assert (k, stride, alloc) == (4, 1024, 3 * 1024 + 1000)
    with pytest.raises(ValueError):
        oracle.rotation_plan(0, 256 << 20)
    with pytest.raises(ValueError):
        oracle.rotation_plan(1 << 62, 2**64 - 1, 0)


def test_slice_for_iteration_folds_negative_warmup():
    assert [oracle.slice_for_iteration(i, 64) for i in (-3, -2, -1, 0, 1, 63, 64, 130)] == \
        [61, 62, 63, 0, 1, 63, 0, 2]
    assert all(oracle.slice_for_iteration(i, 1) == 0 for i in range(-5, 5))
    assert oracle.slice_for_iteration(-64, 64) == 0
    assert oracle.slice_for_iteration(-65, 64) == 63


# ---------------------------------------------------------------------------
# Batch apply - Mooncake RFC "Design of #5040"; compare - ValidateAllTransfers
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(6))
def test_apply_batch_matches_byte_slicing(seed):
    g = np.random.default_rng(seed)
    src = g.integers(0, 256, 4096, dtype=np.uint8)
    dst = g.integers(0, 256, 4096, dtype=np.uint8)
    n = int(g.integers(1, 40))
    lens = g.integers(0, 300, n)
    # non-overlapping destinations: one per 4096/n stretch
    span = 4096 // n
    dst_off = np.array([j * span + int(g.integers(0, max(1, span - lens[j] + 1)))
                        for j in range(n)])
    lens = np.minimum(lens, span - (dst_off - np.arange(n) * span))
    src_off = g.integers(0, 4096 - lens + 1)
    ref = bytearray(dst.tobytes())
    for s, d, ln in zip(src_off, dst_off, lens):
        ref[d:d + ln] = src.tobytes()[s:s + ln]
    out = dst.copy()
    oracle.apply_batch(out, src, src_off, dst_off, lens)
    assert out.tobytes() == bytes(ref)


def test_apply_batch_rejects_out_of_pool():
    src = np.zeros(100, np.uint8)
    dst = np.zeros(100, np.uint8)
    with pytest.raises(ValueError):
        oracle.apply_batch(dst, src, [90], [0], [11])
    with pytest.raises(ValueError):
        oracle.apply_batch(dst, src, [0], [95], [6])
    oracle.apply_batch(dst, src, [0], [0], [100])


def test_first_mismatch_brute_force():
    g = np.random.default_rng(3)
    for _ in range(50):
        a = g.integers(0, 2**32, 257, dtype=np.uint64).astype(np.uint32)
        b = a.copy()
        if g.random() < 0.8:
            idx = g.integers(0, 257, int(g.integers(1, 4)))
            b[idx] ^= np.uint32(1) << np.uint32(g.integers(0, 32))
        diff = np.nonzero(a != b)[0]
        want = int(diff[0]) if diff.size else -1
        assert oracle.first_mismatch(a, b) == want
        assert oracle.first_mismatch(a.view(np.uint8), b.view(np.uint8)) == \
            (int(np.nonzero(a.view(np.uint8) != b.view(np.uint8))[0][0]) if diff.size else -1)
