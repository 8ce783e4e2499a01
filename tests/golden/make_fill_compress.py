"""Writes fill_compress.txt: hand-checkable expected words of fillCompress.

Stand-alone on purpose: plain Python integers only - no numpy, no float
arithmetic, nothing imported from the oracle or the library - so that the
expected words do not come from the code they check.

The reading it follows ("TransferBench data validation", section "Expected
source pattern", fillCompress row, which names modes 0 = random, 1B0, 2B0,
4B0 and 32B0 and says percentages set the mix, but defines neither the masks
nor the random source):
  - buffer k draws from the SplitMix64 stream seeded with seed + k (Steele,
    Lea & Flood, OOPSLA 2014; the published known-answer vector for seed
    1234567 sits in splitmix64.txt and is checked below before anything is
    written);
  - each 64-byte line (16 floats) takes 17 draws in order: the first picks
    the mode, the next 16 give the floats;
  - mode = the first m with (draw % 100) < pct[0] + ... + pct[m];
  - float = (draw >> 40) * 2^-23 - 1, i.e. (m - 2^23) / 2^23 for the 24-bit
    integer m = draw >> 40, exactly representable; its binary32 bits are
    built here from sign, exponent and mantissa by integer arithmetic;
  - mode nB0 zeroes every odd-numbered aligned n-byte chunk of the line, in
    little-endian memory order: per 32-bit word, 1B0 keeps bytes 0 and 2
    (mask 0x00FF00FF), 2B0 keeps bytes 0-1 (mask 0x0000FFFF), 4B0 zeroes
    the odd words, 32B0 zeroes words 8..15;
  - a partial last line keeps its first n % 16 floats.

Run from the repository root:  python tests/golden/make_fill_compress.py
"""
import os

M64 = (1 << 64) - 1
HERE = os.path.dirname(os.path.abspath(__file__))


def splitmix64(seed, count):
    s, out = seed & M64, []
    for _ in range(count):
        s = (s + 0x9E3779B97F4A7C15) & M64
        z = s
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        out.append(z ^ (z >> 31))
    return out


def float_bits(m):
    """binary32 bits of (m - 2^23) / 2^23 for an integer 0 <= m < 2^24."""
    a = m - (1 << 23)
    if a == 0:
        return 0
    sign = 1 if a < 0 else 0
    a = abs(a)                   # 1 <= a <= 2^23, value a * 2^-23
    e = a.bit_length() - 1       # a = 2^e * (1 + f)
    mant = (a - (1 << e)) << (23 - e)
    return (sign << 31) | ((e - 23 + 127) << 23) | mant


MASK_KEEP = {1: 0x00FF00FF, 2: 0x0000FFFF}


def masked(words, mode):
    out = list(words)
    for j in range(16):
        if mode in MASK_KEEP:
            out[j] &= MASK_KEEP[mode]
        elif mode == 3 and j % 2 == 1:
            out[j] = 0
        elif mode == 4 and j >= 8:
            out[j] = 0
    return out


def expected(n, pct, seed, k):
    lines = (n + 15) // 16
    draws = splitmix64(seed + k, 17 * lines)
    cum = [sum(pct[:m + 1]) for m in range(5)]
    out, modes = [], []
    for line in range(lines):
        d = draws[17 * line: 17 * line + 17]
        r = d[0] % 100
        mode = next(m for m in range(5) if r < cum[m])
        modes.append(mode)
        words = masked([float_bits(x >> 40) for x in d[1:]], mode)
        out.extend(words)
    return out[:n], modes


# (name, seed, k, n, percentages): line 0 of seed 1234567 draws r = 17 and
# line 1 draws r = 99, so these percentages put every mode on a full line
# and several on the partial second line, with r equal to a running sum in
# two of them (a line whose r equals the sum goes to the next mode).
CASES = [
    ("random_then_32B0", 1234567, 0, 21, (18, 0, 0, 0, 82)),
    ("1B0_at_boundary", 1234567, 0, 21, (17, 83, 0, 0, 0)),
    ("2B0_both", 1234567, 0, 21, (0, 0, 100, 0, 0)),
    ("4B0_then_32B0", 1234567, 0, 21, (10, 0, 0, 8, 82)),
    ("32B0_at_boundary", 1234567, 0, 21, (10, 0, 0, 7, 83)),
    ("4B0_both", 1234567, 0, 21, (0, 0, 0, 100, 0)),
    ("seed_plus_k", 1234559, 8, 21, (18, 0, 0, 0, 82)),
    ("one_partial_line", 1234567, 0, 5, (0, 100, 0, 0, 0)),
]


def check_published_vector():
    rows = []
    with open(os.path.join(HERE, "splitmix64.txt")) as f:
        for line in f:
            t = line.split()
            if t and not line.startswith("#") and t[0] != "counts":
                rows.append(t)
    got = splitmix64(int(rows[0][0]), len(rows))
    for seed, idx, val in rows:
        assert got[int(idx)] == int(val), (seed, idx)


HEADER = """\
# fillCompress, hand-checkable expected words ("TransferBench data validation",
# section "Expected source pattern", fillCompress row), written by
# make_fill_compress.py in this folder (plain Python integers, nothing imported).
#
# Reading: buffer k draws SplitMix64 seeded with seed + k; per 64-byte line the
# first draw d0 gives the mode (first m with d0 % 100 < pct[0] + .. + pct[m]),
# the next 16 give the floats (d >> 40) * 2^-23 - 1; mode nB0 zeroes every
# odd-numbered aligned n-byte chunk of the line (little-endian).
#
# Derivation by hand of the first float of seed 1234567, line 0:
#   d1 = 3203168211198807973 (published vector, index 1)
#   m = d1 >> 40 = 2913264; m - 2^23 = -5475344, value -5475344 / 2^23
#   5475344 = 2^22 * 1.30542755..., so exponent 22 - 23 = -1 (biased 126),
#   mantissa (5475344 - 2^22) * 2 = 2562080 = 0x271820, sign 1
#   bits = 0x80000000 | 126 << 23 | 0x271820 = 0xBF271820
# Mode of line 0: d0 = 6457827717110365317, d0 % 100 = 17; of line 1:
#   d17 % 100 = 99.
# Masks per 32-bit word: 1B0 & 0x00FF00FF, 2B0 & 0x0000FFFF, 4B0 odd words
# -> 0, 32B0 words 8..15 -> 0.
#
# Row kinds:
#   draw  <stream seed> <index> <value> <value % 100> <value >> 40>
#   case  <name> <seed> <k> <n> <pct0> <pct1> <pct2> <pct3> <pct4> <mode of each line...>
#   word  <name> <index> <bits, hex>
"""


def main():
    check_published_vector()
    lines = [HEADER]
    for i, v in enumerate(splitmix64(1234567, 34)):
        lines.append(f"draw 1234567 {i} {v} {v % 100} {v >> 40}\n")
    for name, seed, k, n, pct in CASES:
        words, modes = expected(n, pct, seed, k)
        lines.append(f"case {name} {seed} {k} {n} " + " ".join(map(str, pct)) + " "
                     + " ".join(map(str, modes)) + "\n")
        for i, w in enumerate(words):
            lines.append(f"word {name} {i} {w:08X}\n")
    with open(os.path.join(HERE, "fill_compress.txt"), "w") as f:
        f.writelines(lines)


if __name__ == "__main__":
    main()
