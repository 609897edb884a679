"""Write int8_quotient.txt and q4_quotient.txt: quantiser inputs whose codes
depend on HOW the quotient is rounded.

The k8v4 PR (Tests section: int8 codes round half to even; What section: V
stored as rotated q4_0) fixes the rounding of the code but not the arithmetic
of the quotient.
This library reads it as ONE IEEE fp32 division, x / s (int8 K) and y / d
(q4_0 V), each correctly rounded, then rint ties-to-even.  Two plausible
alternatives give different codes on some inputs:
  - multiplying by the rounded reciprocal: RN(x * RN(1 / s));
  - (int8 only) dividing the scaled value by the absmax: RN(RN(x * 127) / a).
This script finds such inputs with exact rational arithmetic only (Python
Fractions; no floating-point division, no oracle, no GPU) and records, per
case, the exact quotient, its fp32 rounding and the code each reading gives,
so a reader can check every line by hand.

Run from the repository root:  python tests/golden/make_quotient_cases.py
"""
from __future__ import annotations

import os
import random
from fractions import Fraction

HERE = os.path.dirname(os.path.abspath(__file__))


def round_binary(v: Fraction, mant_bits: int, emin: int, emax: int) -> Fraction:
    """Round v to the nearest number with `mant_bits` significand bits
    (including the leading one), exponent >= emin (subnormals below), ties to
    even; overflow gives None."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, emin)
    ulp = Fraction(2) ** (e - mant_bits + 1)
    q, r = divmod(a, ulp)
    q = int(q)
    if r * 2 > ulp or (r * 2 == ulp and q % 2 == 1):
        q += 1
    res = q * ulp
    if res >= Fraction(2) ** (emax + 1):
        return None
    return sign * res


def rn32(v: Fraction) -> Fraction:
    return round_binary(v, 24, -126, 127)


def rn16(v: Fraction) -> Fraction:
    return round_binary(v, 11, -14, 15)


def rint_even(v: Fraction) -> int:
    f = v.numerator // v.denominator
    r = v - f
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return int(f)


def hexf(v: Fraction) -> str:
    return float(v).hex()


def ulp_of(v: Fraction) -> Fraction:
    """Spacing of fp32 numbers at the normal value v."""
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    return Fraction(2) ** (e - 23)


def int8_code(q: Fraction) -> int:
    return max(-127, min(127, rint_even(q)))


def int8_cases(rng: random.Random, want: int = 6):
    """(a, x) with a = the half's absmax (lane 0), x at lane 1."""
    by_recip, by_a = [], []
    seen = set()
    tries = 0
    while (len(by_recip) < want or len(by_a) < want) and tries < 200000:
        tries += 1
        sig = rng.randrange(1 << 23, 1 << 24)
        if sig & (sig - 1) == 0:
            continue
        a = Fraction(sig, 1 << 23) * Fraction(2) ** rng.randrange(-6, 7)
        s = rn32(a / 127)
        k = rng.randrange(-127, 127)
        x0 = rn32((Fraction(2 * k + 1, 2)) * s)
        for j in (-2, -1, 0, 1, 2):
            x = rn32(x0 + j * ulp_of(x0))
            if x == 0 or abs(x) >= a or x in seen:
                continue
            seen.add(x)
            q_true = rn32(x / s)
            q_rec = rn32(x * rn32(1 / s))
            q_a = rn32(rn32(x * 127) / a)
            c_true, c_rec, c_a = int8_code(q_true), int8_code(q_rec), int8_code(q_a)
            row = (a, s, x, q_true, c_true, q_rec, c_rec, q_a, c_a)
            if c_rec != c_true and len(by_recip) < want:
                by_recip.append(row)
            elif c_a != c_true and len(by_a) < want:
                by_a.append(row)
    return by_recip + by_a


def q4_code(q: Fraction) -> int:
    return max(0, min(15, rint_even(q) + 8))


def q4_cases(rng: random.Random, want: int = 8):
    """(m, y) with m the block's extreme (lane 0) and y at lane 1."""
    out = []
    seen = set()
    tries = 0
    while len(out) < want and tries < 400000:
        tries += 1
        sig = rng.randrange(1 << 10, 1 << 11)          # d = fp16 with a non-power-of-two significand
        if sig & (sig - 1) == 0:
            continue
        d = -Fraction(sig, 1 << 10) * Fraction(2) ** rng.randrange(-4, 4) * rng.choice((1, -1))
        m = rn32(-8 * d)                               # exact: m / -8 = d, fp16_RN(d) = d
        assert rn16(m / -8) == d
        k = rng.randrange(-8, 7)
        y0 = rn32(Fraction(2 * k + 1, 2) * d)
        for j in (-2, -1, 0, 1, 2):
            y = rn32(y0 + j * ulp_of(y0))
            if y == 0 or abs(y) >= abs(m) or y in seen:
                continue
            seen.add(y)
            q_true = rn32(y / d)
            q_rec = rn32(y * rn32(1 / d))
            c_true, c_rec = q4_code(q_true), q4_code(q_rec)
            if c_rec != c_true:
                out.append((m, d, y, q_true, c_true, q_rec, c_rec))
                break
    return out


def main():
    rng = random.Random(0x6B38763451)
    rows = int8_cases(rng)
    with open(os.path.join(HERE, "int8_quotient.txt"), "w") as f:
        f.write("# int8 K codes that depend on the quotient's arithmetic (written by\n"
                "# make_quotient_cases.py with exact rational arithmetic).  The half's lane 0\n"
                "# holds the absmax a, lane 1 holds x, all other lanes 0.\n"
                "#   s = RN32(a / 127); code = clamp(rint_even(RN32(x / s)), -127, 127)  (this library)\n"
                "#   reciprocal reading:  RN32(x * RN32(1 / s))\n"
                "#   absmax reading:      RN32(RN32(x * 127) / a)\n"
                "# Columns: a x s (fp32 hex) | code | RN32(x/s) | reciprocal code, quotient |\n"
                "#          absmax code, quotient.  Values are exact (float.hex of fp32).\n")
        for a, s, x, q_true, c_true, q_rec, c_rec, q_a, c_a in rows:
            f.write(f"{hexf(a)} {hexf(x)} {hexf(s)} | {c_true} {hexf(q_true)} | {c_rec} {hexf(q_rec)} | "
                    f"{c_a} {hexf(q_a)}\n")
    rows4 = q4_cases(rng)
    with open(os.path.join(HERE, "q4_quotient.txt"), "w") as f:
        f.write("# Q4_0 V codes that depend on the quotient's arithmetic (written by\n"
                "# make_quotient_cases.py with exact rational arithmetic).  One rotated block:\n"
                "# lane 0 holds m (the element of largest |y|), lane 1 holds y, all other lanes 0.\n"
                "#   d = fp16_RN(m / -8) (exact here: m = -8 d); code = clamp(rint_even(RN32(y / d)) + 8, 0, 15)\n"
                "#   reciprocal reading:  RN32(y * RN32(1 / d))\n"
                "# Columns: m y d (hex) | code | RN32(y/d) | reciprocal code, quotient.\n")
        for m, d, y, q_true, c_true, q_rec, c_rec in rows4:
            f.write(f"{hexf(m)} {hexf(y)} {hexf(d)} | {c_true} {hexf(q_true)} | {c_rec} {hexf(q_rec)}\n")
    print(f"{len(rows)} int8 cases, {len(rows4)} q4 cases")


if __name__ == "__main__":
    main()
